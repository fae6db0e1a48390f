// Fused indexer scoring + exact Top-k selection, one thread-block cluster per
// query.
//
// The C CTAs of a cluster split one query's candidate rows: CTA c scores rows
// [c * rows_per_cta, (c + 1) * rows_per_cta) -- a contiguous run of indexer
// keys (flat mode: every valid entry, or every valid block summary key) or the
// entries of a run of pooled blocks (pooled mode) -- exactly like the
// streaming indexer kernel (one producer warp feeding a TMA bulk-copy ring,
// four consumer warps running mma.sync m16n8k16 on q_idx . K^T).  Instead of
// writing the scores to global memory, each CTA keeps their order keys in
// shared memory.  The cluster then selects the Top-k under (score descending,
// index ascending) with a distributed radix select: every pass builds a local
// 256-bin histogram (in the now idle ring buffer),
// publishes its totals, and after one cluster barrier every CTA sums the C
// totals through distributed shared memory and keeps the same bin.  Each bin
// has 8 counter copies (one per lane & 7), which keeps the clear and the
// reduction cheap while bounding same-address contention to 4 lanes.  The tie
// quota and output offset of each CTA come from a prefix over the CTAs, and
// because the CTAs hold ascending index ranges the selected ids are written
// directly in ascending order.
//
// (DeepSeek V4.1 Flash architecture page: bullet "Hierarchical indexer" -- block
// pool, at most 16,384 candidates; bullet "Sparse attention" -- Top-512.)
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kHeads = 8;
constexpr int kDim = 64;
constexpr int kRowBytes = kDim * 2;
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kRowBytes;    // 16 KB
constexpr int kStages = 3;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;      // 160
constexpr int kWarpsAll = kThreads / 32;
constexpr int kBlock = 8;
constexpr int kBlockBytes = kBlock * kRowBytes;
constexpr int kBlocksPerTile = kTileRows / kBlock;
constexpr int kBins = 256;
constexpr int kCopies = 8;                           // counter copies per bin (lane & 7)
constexpr int kMaxCluster = 8;
constexpr int kMaxRowsPerCta = 4096;                 // order keys kept in shared memory

static_assert(kBins * kCopies * 4 <= kStages * kTileBytes, "histogram reuses the ring buffer");

struct SelSmall {
  uint32_t tot[2][kBins];
  uint32_t gtot[kBins];
  uint32_t red[3][kWarpsAll];
  uint32_t stats[3];    // this CTA: valid count, min key, max key
  uint32_t fin[2];      // this CTA: count > T, count == T
  uint32_t sel_bin, sel_above, lo, hi, n_valid, offset, quota;
  uint64_t full[kStages];
  uint64_t empty[kStages];
};

constexpr size_t kOffSmall = size_t(kStages) * kTileBytes;
constexpr size_t kOffKeys = kOffSmall + ((sizeof(SelSmall) + 127) / 128) * 128;

size_t select_smem_bytes(int rows_per_cta, bool pooled) {
  const int rows = pooled ? rows_per_cta * kBlock : rows_per_cta;
  return kOffKeys + size_t(rows) * 4 + (pooled ? size_t(rows_per_cta) * 4 : 0);
}

template <bool POOLED>
__global__ void __launch_bounds__(kThreads) index_select_kernel(const SelectArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  SelSmall& sm = *reinterpret_cast<SelSmall*>(smem + kOffSmall);
  uint32_t* s_key = reinterpret_cast<uint32_t*>(smem + kOffKeys);
  const int units_cap = a.rows_per_cta;                                 // rows (flat) or blocks (pooled)
  int* s_pool = reinterpret_cast<int*>(s_key + (POOLED ? units_cap * kBlock : units_cap));
  uint32_t(*hist)[kCopies] = reinterpret_cast<uint32_t(*)[kCopies]>(smem);   // after scoring

  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank(), ncta = cluster_size();
  pdl_launch_dependents();

  const int nv = clamp_count(a.n_valid[b], a.valid_cap, a.err);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumers);
    }
    mbar_fence_init();
  }
  pdl_wait();   // the pool / n_pool come from the preceding launch

  // ---------------- this CTA's share of the query's candidates
  int n_units;
  if (!POOLED)
    n_units = (nv + a.div - 1) / a.div;
  else
    n_units = clamp_count(a.n_pool[b], a.pool_cap, a.err);
  const int begin = int(crank) * units_cap;
  const int end = min(begin + units_cap, n_units);
  const int n_loc_units = max(0, end - begin);
  const int rows_total = POOLED ? n_loc_units * kBlock : n_loc_units;
  const int nb_valid = (nv + kBlock - 1) / kBlock;
  if (POOLED) {
    for (int i = tid; i < n_loc_units; i += kThreads) {
      int blk = a.pool[(long long)b * a.pool_cap + begin + i];
      if (blk < 0 || blk >= nb_valid) {
        report(a.err, kErrBadPool, blk);
        blk = -1;
      }
      s_pool[i] = blk;
    }
  }
  __syncthreads();

  // ---------------- phase 1: stream and score (keys -> s_key)
  uint32_t my_cnt = 0u, my_lo = 0xffffffffu, my_hi = 0u;   // this thread's keys
  const int ntiles = (rows_total + kTileRows - 1) / kTileRows;
  const uint8_t* keys = static_cast<const uint8_t*>(a.keys) + (long long)b * a.rows_per_seq * kRowBytes;
  if (warp == kConsumers) {
    int i = 0;
    for (; i < ntiles; ++i) {
      const int s = i % kStages;
      bool ok = true;
      if (lane == 0 && i >= kStages) ok = mbar_wait(&sm.empty[s], ((i / kStages) - 1) & 1);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* dst = tiles + s * kTileBytes;
      if (!POOLED) {
        if (lane == 0) {
          const int r0 = begin + i * kTileRows;
          const uint32_t bytes = uint32_t(min(kTileRows, end - r0)) * kRowBytes;
          mbar_arrive_expect_tx(&sm.full[s], bytes);
          bulk_g2s(dst, keys + (long long)r0 * kRowBytes, bytes, &sm.full[s]);
        }
      } else {
        const int p0 = i * kBlocksPerTile;
        const int np = min(kBlocksPerTile, n_loc_units - p0);
        const int blk = lane < np ? s_pool[p0 + lane] : -1;
        const unsigned have = __ballot_sync(0xffffffffu, blk >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], uint32_t(__popc(have)) * kBlockBytes);
        __syncwarp();
        if (blk >= 0)
          bulk_g2s(dst + lane * kBlockBytes, keys + (long long)blk * kBlockBytes, kBlockBytes, &sm.full[s]);
      }
    }
    if (lane == 0) {
      if (i < ntiles) report(a.err, kErrTimeout, i);
      for (int j = max(0, i - kStages); j < i; ++j) mbar_wait(&sm.full[j % kStages], (j / kStages) & 1);
    }
  } else {
    const int g = lane >> 2, t = lane & 3;
    const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q_idx) +
                                                     (((long long)b * kHeads + g) * kDim + 16 * t) * 2);
    const uint4 q0 = qp[0], q1 = qp[1];
    const uint32_t qf[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const float w0 = a.w[b * kHeads + 2 * t];
    const float w1 = a.w[b * kHeads + 2 * t + 1];
    const bool relu = a.relu != 0;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kStages;
      if (!mbar_wait(&sm.full[s], (i / kStages) & 1)) {
        report(a.err, kErrTimeout, i);
        break;
      }
      const uint8_t* tile = tiles + s * kTileBytes;
      (void)tile;
      uint32_t ra[2][8], rb[2][8];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint8_t* p = tile + ((warp * 2 + m) * 16 + g) * kRowBytes + 32 * t;
        const uint4 x0 = *reinterpret_cast<const uint4*>(p);
        const uint4 x1 = *reinterpret_cast<const uint4*>(p + 16);
        const uint4 y0 = *reinterpret_cast<const uint4*>(p + 8 * kRowBytes);
        const uint4 y1 = *reinterpret_cast<const uint4*>(p + 8 * kRowBytes + 16);
        ra[m][0] = x0.x; ra[m][1] = x0.y; ra[m][2] = x0.z; ra[m][3] = x0.w;
        ra[m][4] = x1.x; ra[m][5] = x1.y; ra[m][6] = x1.z; ra[m][7] = x1.w;
        rb[m][0] = y0.x; rb[m][1] = y0.y; rb[m][2] = y0.z; rb[m][3] = y0.w;
        rb[m][4] = y1.x; rb[m][5] = y1.y; rb[m][6] = y1.z; rb[m][7] = y1.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16(c0, ra[m][0], rb[m][0], ra[m][1], rb[m][1], qf[0], qf[1]);
        mma_bf16(c1, ra[m][2], rb[m][2], ra[m][3], rb[m][3], qf[2], qf[3]);
        mma_bf16(c0, ra[m][4], rb[m][4], ra[m][5], rb[m][5], qf[4], qf[5]);
        mma_bf16(c1, ra[m][6], rb[m][6], ra[m][7], rb[m][7], qf[6], qf[7]);
        float h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float d = c0[e] + c1[e];
          h[e] = relu ? fmaxf(d, 0.f) : d;
        }
        float r0 = __fadd_rn(__fmul_rn(w0, h[0]), __fmul_rn(w1, h[1]));
        float r1 = __fadd_rn(__fmul_rn(w0, h[2]), __fmul_rn(w1, h[3]));
        r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
        r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
        r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
        r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
        const int row = i * kTileRows + (warp * 2 + m) * 16 + g + 8 * t;
        if (t < 2 && row < rows_total) {
          bool valid = true;
          if (POOLED) {
            const int blk = s_pool[row / kBlock];
            valid = blk >= 0 && blk * kBlock + row % kBlock < nv;
          }
          const uint32_t kk = valid ? score_key(t == 0 ? r0 : r1) : 0u;   // 0: not a candidate
          s_key[row] = kk;
          if (kk != 0u) {
            ++my_cnt;
            my_lo = min(my_lo, kk);
            my_hi = max(my_hi, kk);
          }
        }
      }
    }
  }
  __syncthreads();   // all keys written; the ring buffer is free for the histogram

  // ---------------- phase 2: cluster-wide exact Top-k over the keys
  // (count, min, max) of the keys, tracked while scoring
  {
    uint32_t cnt = my_cnt, lo = my_lo, hi = my_hi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      sm.red[0][warp] = cnt;
      sm.red[1][warp] = lo;
      sm.red[2][warp] = hi;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t c = 0, l = 0xffffffffu, h = 0u;
      for (int w = 0; w < kWarpsAll; ++w) {
        c += sm.red[0][w];
        l = min(l, sm.red[1][w]);
        h = max(h, sm.red[2][w]);
      }
      sm.stats[0] = c;
      sm.stats[1] = l;
      sm.stats[2] = h;
    }
    cluster_sync_all();
    if (tid == 0) {
      uint32_t rc[kMaxCluster], rl[kMaxCluster], rh[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < int(ncta)) {
          rc[r] = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.stats[0], r)));
          rl[r] = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.stats[1], r)));
          rh[r] = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.stats[2], r)));
        } else {
          rc[r] = 0u;
          rl[r] = 0xffffffffu;
          rh[r] = 0u;
        }
      }
      uint32_t c = 0, l = 0xffffffffu, h = 0u;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        c += rc[r];
        if (rc[r] > 0) {
          l = min(l, rl[r]);
          h = max(h, rh[r]);
        }
      }
      sm.n_valid = c;
      sm.lo = l;
      sm.hi = h;
    }
    __syncthreads();
  }
  const uint32_t n_sel_valid = sm.n_valid;
  const uint32_t k = uint32_t(a.k);
  const bool take_all = n_sel_valid <= k;
  uint32_t T = 0u, need_eq = 0u;
  if (!take_all) {
    uint32_t lo = sm.lo, hi = sm.hi, above = 0u;
    int buf = 0;
    while (lo != hi) {
      const uint32_t range = hi - lo;
      const int bits = 32 - __clz(range);
      const int shift = bits > 8 ? bits - 8 : 0;
      uint4* hv = reinterpret_cast<uint4*>(&hist[0][0]);
      for (int j = tid; j < kBins * kCopies / 4; j += kThreads) hv[j] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      for (int j0 = tid; j0 < rows_total; j0 += 8 * kThreads) {
        uint32_t kk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) kk[u] = j0 + u * kThreads < rows_total ? s_key[j0 + u * kThreads] : 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (kk[u] != 0u && kk[u] >= lo && kk[u] <= hi)
            atomicAdd(&hist[(kk[u] - lo) >> shift][lane & (kCopies - 1)], 1u);
      }
      __syncthreads();
      for (int bin = tid; bin < kBins; bin += kThreads) {
        const uint4 x = *reinterpret_cast<const uint4*>(&hist[bin][0]);
        const uint4 y = *reinterpret_cast<const uint4*>(&hist[bin][4]);
        sm.tot[buf][bin] = x.x + x.y + x.z + x.w + y.x + y.y + y.z + y.w;
      }
      cluster_sync_all();
      for (int bin = tid; bin < kBins; bin += kThreads) {
        uint32_t rv[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          rv[r] = r < int(ncta) ? __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.tot[buf][bin], r))) : 0u;
        uint32_t v = 0u;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) v += rv[r];
        sm.gtot[bin] = v;
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

  // ---------------- phase 3: this CTA's quota, offset and ordered output
  // Each thread owns a contiguous run of local positions so that a block scan
  // in thread order is a scan in position order.
  const int per_thread = (rows_total + kThreads - 1) / kThreads;
  const int r0 = min(rows_total, tid * per_thread);
  const int r1 = min(rows_total, r0 + per_thread);
  uint32_t n_gt = 0u, n_eq = 0u;
  for (int j0 = r0; j0 < r1; j0 += 8) {
    uint32_t kk[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) kk[u] = j0 + u < r1 ? s_key[j0 + u] : 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (kk[u] == 0u) continue;
      if (take_all || kk[u] > T)
        ++n_gt;
      else if (kk[u] == T)
        ++n_eq;
    }
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
      for (int w = 0; w < kWarpsAll; ++w) {
        gg += sm.red[0][w];
        ee += sm.red[1][w];
      }
      sm.fin[0] = gg;
      sm.fin[1] = ee;
    }
    cluster_sync_all();
    if (tid == 0) {
      uint32_t rg[kMaxCluster], re[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        rg[r] = r < int(crank) ? __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.fin[0], r))) : 0u;
        re[r] = r < int(crank) ? __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.fin[1], r))) : 0u;
      }
      uint32_t off = 0, eq_before = 0;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        off += rg[r] + min(re[r], need_eq > eq_before ? need_eq - eq_before : 0u);
        eq_before += re[r];
      }
      sm.offset = off;
      sm.quota = min(sm.fin[1], need_eq > eq_before ? need_eq - eq_before : 0u);
    }
    __syncthreads();
  }
  // exclusive block scan of (n_gt << 16 | n_eq) in thread order
  uint32_t gt_before, eq_before;
  {
    const uint32_t v = (n_gt << 16) | n_eq;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm.red[2][warp] = x;
    __syncthreads();
    uint32_t pre = 0u;
    for (int w = 0; w < warp; ++w) pre += sm.red[2][w];
    const uint32_t ex = pre + x - v;
    gt_before = ex >> 16;
    eq_before = ex & 0xffffu;
  }
  const uint32_t quota = sm.quota;
  uint32_t slot = sm.offset + gt_before + min(eq_before, quota);
  int* out = a.out + (long long)b * a.ld_out;
  for (int j0 = r0; j0 < r1; j0 += 8) {
    uint32_t kk[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) kk[u] = j0 + u < r1 ? s_key[j0 + u] : 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (kk[u] == 0u) continue;
      bool take = false;
      if (take_all || kk[u] > T) {
        take = true;
      } else if (kk[u] == T) {
        take = eq_before < quota;
        ++eq_before;
      }
      if (take) {
        const int j = j0 + u;
        int id;
        if (!POOLED)
          id = begin + j;
        else
          id = s_pool[j / kBlock] * kBlock + j % kBlock;
        out[slot++] = id;
      }
    }
  }
  const int selected = int(min(n_sel_valid, k));
  if (crank == 0) {
    if (a.n_out != nullptr && tid == 0) a.n_out[b] = selected;
    for (int j = selected + tid; j < a.k; j += kThreads) out[j] = -1;
  }
  cluster_sync_all();   // no CTA leaves while another may still read its shared memory
}

struct ClusterChoice {
  int c = 0;
  int units_per_cta = 0;
  size_t smem = 0;
};

}  // namespace

// Choose the cluster size: enough CTAs that a CTA's rows fit in shared memory,
// as many as keep every cluster of the batch resident at once (one wave).
static cudaError_t choose(bool pooled, int max_units, int batch, ClusterChoice& out) {
  const int unit_rows = pooled ? kBlock : 1;
  auto kern = pooled ? index_select_kernel<true> : index_select_kernel<false>;
  ClusterChoice best;
  for (int c = kMaxCluster; c >= 1; --c) {
    const int per = (max_units + c - 1) / c;
    if (per * unit_rows > kMaxRowsPerCta) break;
    const size_t smem = select_smem_bytes(per, pooled);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(c), unsigned(batch), 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (best.c == 0) best = ClusterChoice{c, per, smem};
    if (active >= batch) {
      out = ClusterChoice{c, per, smem};
      return cudaSuccess;
    }
  }
  out = best;
  return cudaSuccess;
}

bool index_select_supported(bool pooled, int max_units) {
  const int unit_rows = pooled ? kBlock : 1;
  return (max_units + kMaxCluster - 1) / kMaxCluster * unit_rows <= kMaxRowsPerCta;
}

cudaError_t launch_index_select(const SelectArgs& in, bool pooled, int batch, int max_units, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  // the occupancy query is made once per (device, mode, size, batch)
  struct Entry {
    int dev, pooled, units, batch;
    ClusterChoice ch;
  };
  static Entry cache[16];
  static int n_cache = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  ClusterChoice ch;
  bool hit = false;
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].dev == dev && cache[i].pooled == int(pooled) && cache[i].units == max_units &&
        cache[i].batch == batch) {
      ch = cache[i].ch;
      hit = true;
    }
  cudaError_t e = cudaSuccess;
  if (!hit) {
    e = choose(pooled, max_units, batch, ch);
    if (e != cudaSuccess) return e;
    cache[n_cache % 16] = Entry{dev, int(pooled), max_units, batch, ch};
    ++n_cache;
  }
  if (ch.c == 0) return cudaErrorInvalidValue;
  SelectArgs a = in;
  a.rows_per_cta = ch.units_per_cta;
  auto kern = pooled ? index_select_kernel<true> : index_select_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(ch.smem));
  if (e != cudaSuccess) return e;
  note_launch();
  return launch_pdl(kern, dim3(unsigned(ch.c), unsigned(batch), 1), dim3(kThreads), ch.smem, st, unsigned(ch.c), a);
}

}  // namespace csa2

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
// shared memory and the cluster selects the Top-k under (score descending,
// index ascending) with three cluster barriers in the common case:
//
//   1. every CTA pushes (count, min, max) of its keys into every CTA;
//   2. a radix pass: every CTA histograms its keys into 256 bins over the
//      common [min, max] range and pushes the bin totals into every CTA, so
//      that after the barrier each CTA holds all C histograms and finds the
//      bin holding the k-th key, the keys above it, and each CTA's share of
//      both;
//   3. every CTA pushes its keys inside that bin into every CTA, which then
//      finishes the selection alone (passes over the gathered keys, each
//      narrowing to the exact [min, max] of the chosen bin) and counts each
//      CTA's keys above and at the threshold.  The radix pass stores each
//      key's bin as a byte, so finding the keys of the chosen bin compares
//      bytes instead of binning every key again.
//
// Only while the chosen bin holds more keys than a CTA can gather do steps 1
// and 2 repeat on the keys of that bin.  The first pass of each loop bins the
// score values linearly between the range's end points (a monotone map, so
// every bin is a contiguous key range); later passes bin the order-key bits,
// which removes at least 8 bits of the range per pass.
//
// All remote traffic is stores into the destination's shared memory, so no
// step waits on a remote load.  Ties at the threshold go to the lowest
// indices: the CTAs hold ascending index ranges, so each CTA's quota and
// output offset follow from the per-CTA counts, and each CTA writes its ids
// directly in ascending order (one pass lists each warp's keys at or above the
// threshold, a second writes the ids from those short lists).
//
// (DeepSeek V4.1 Flash architecture page: bullet "Hierarchical indexer" -- block
// pool, at most 16,384 candidates; bullet "Sparse attention" -- Top-512.)
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kHeads = 8;
constexpr int kDim = 64;
constexpr int kRowBytes = kDim * 2;
constexpr int kTileRows = 64;
constexpr int kTileBytes = kTileRows * kRowBytes;    // 8 KB
constexpr int kStages = 5;
constexpr int kConsumers = 4;
constexpr int kMTiles = kTileRows / 16 / kConsumers; // 16-row MMA tiles per consumer warp and tile
static_assert(kTileRows == 16 * kMTiles * kConsumers, "consumer warps split a tile evenly");
constexpr int kThreads = (kConsumers + 1) * 32;      // 160
constexpr int kWarpsAll = kThreads / 32;
constexpr int kBlock = 8;
constexpr int kBlockBytes = kBlock * kRowBytes;
constexpr int kBlocksPerTile = kTileRows / kBlock;
constexpr int kBins = 256;
constexpr int kMaxCluster = 16;                       // 16 is a non-portable cluster size (small batches only)
constexpr int kPortableCluster = 8;
constexpr int kMaxRowsPerCta = 4096;                 // order keys kept in shared memory
constexpr int kMaxRowsPerCta16 = 2048;               // with more than 8 CTAs: the cluster's keys stay < 65,536
// After scoring, the ring buffer is reused:
//   region A: the histogram of a cluster-wide pass, two bins per word (16-bit
//             counters, 16 copies shared by lanes l and l + 16), then the gather buffer;
//             its tail first holds the bin of every key of the last pass (one
//             byte per key, so that later tests need no binning), then the
//             histogram (kCopiesL copies) and totals of the passes over the
//             gathered keys;
//   region B: the per-CTA bin totals pushed by every CTA, 16-bit counts two
//             bins per word, in two buffers.
constexpr int kRingWords = kStages * kTileBytes / 4;
constexpr int kLanes = 16;                           // histogram copies: lanes l and l + 16 share one
constexpr int kHistDWords = (kBins / 2) * kLanes;
constexpr int kTotWords = kMaxCluster * kBins / 2;                  // one totals buffer
constexpr int kRegionA = kRingWords - 2 * kTotWords;
constexpr int kCopiesL = 8;
constexpr int kLocalWords = kBins * kCopiesL + kBins;               // local histogram + totals
constexpr int kBinWords = kMaxRowsPerCta / 4;
constexpr int kGatherWords = kRegionA - kLocalWords;                // gather buffer capacity

static_assert(kHistDWords <= kGatherWords, "histogram fits region A below its tail");
static_assert(kBinWords <= kLocalWords, "key bins fit the tail of region A");
static_assert(kGatherWords % 4 == 0, "16-byte aligned tail");
static_assert(kMaxRowsPerCta < 65536, "16-bit histogram counters");

struct SelSmall {
  uint4 stats[kMaxCluster];        // pushed by every CTA: (keys, min key, max key, 0)
  uint32_t red[3][kWarpsAll];
  uint32_t above_r[kMaxCluster];   // per CTA: keys above the current range
  uint32_t cnt_r[kMaxCluster];     // per CTA: keys inside the current range
  uint32_t gt_r[kMaxCluster];      // per CTA: keys above the threshold
  uint32_t eq_r[kMaxCluster];      // per CTA: keys at the threshold
  uint32_t gt_g[kMaxCluster];      // rank finish: per CTA, gathered keys above / at the threshold
  uint32_t eq_g[kMaxCluster];
  uint32_t sel_bin, sel_above, gcount;
  uint32_t failed;                 // a bounded wait of this CTA gave up
  uint64_t full[kStages];
  uint64_t empty[kStages];
};

// A monotone map of the order keys inside [lo, hi] to kBins bins: either
// linear in the score value (first passes) or the top bits of (key - lo).
struct Binning {
  uint32_t lo;
  int shift;
  float vlo, scale;
  bool lin;
};

__device__ __forceinline__ Binning make_binning(uint32_t lo, uint32_t hi, bool allow_linear) {
  Binning bn;
  bn.lo = lo;
  const int bits = 32 - __clz(hi - lo);
  bn.shift = bits > 8 ? bits - 8 : 0;
  bn.lin = false;
  bn.vlo = 0.f;
  bn.scale = 0.f;
  if (allow_linear) {
    const float x = key_score(lo), y = key_score(hi);
    const float d = __fsub_rn(y, x);
    if (isfinite(x) && isfinite(y) && isfinite(d) && d > 0.f) {
      const float sc = __fdiv_rn(float(kBins), d);
      if (isfinite(sc) && sc > 0.f) {
        bn.lin = true;
        bn.vlo = x;
        bn.scale = sc;
      }
    }
  }
  return bn;
}

// Bin of a key inside [lo, hi]: non-decreasing in the key, 0 at lo.
__device__ __forceinline__ uint32_t bin_of(uint32_t key, const Binning& bn) {
  if (bn.lin) {
    const float x = __fmul_rn(__fsub_rn(key_score(key), bn.vlo), bn.scale);
    return min(uint32_t(kBins - 1), __float2uint_rz(x));
  }
  return (key - bn.lo) >> bn.shift;
}

// Keys 4i .. 4i + 3 and 4(i + kThreads) .. 4(i + kThreads) + 3 of a key array of
// nvec 16-byte vectors (i < nvec; zeros past the end).
__device__ __forceinline__ void load_keys8(const uint4* kv, int i, int nvec, uint32_t (&kk)[8]) {
  const uint4 x = kv[i];
  const uint4 y = i + kThreads < nvec ? kv[i + kThreads] : make_uint4(0u, 0u, 0u, 0u);
  kk[0] = x.x;
  kk[1] = x.y;
  kk[2] = x.z;
  kk[3] = x.w;
  kk[4] = y.x;
  kk[5] = y.y;
  kk[6] = y.z;
  kk[7] = y.w;
}

constexpr size_t kOffSmall = size_t(kStages) * kTileBytes;
constexpr size_t kOffKeys = kOffSmall + ((sizeof(SelSmall) + 127) / 128) * 128;

// Keys are stored in a multiple of 4 words so that 16-byte reads stay inside them.
__host__ __device__ constexpr int key_words(int rows) { return (rows + 3) & ~3; }

size_t select_smem_bytes(int rows_per_cta, bool pooled) {
  const int rows = pooled ? rows_per_cta * kBlock : rows_per_cta;
  return kOffKeys + size_t(key_words(rows)) * 4 + (pooled ? size_t(rows_per_cta) * 4 : 0);
}

template <bool POOLED>
__global__ void __launch_bounds__(kThreads, 4) index_select_kernel(const SelectArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  SelSmall& sm = *reinterpret_cast<SelSmall*>(smem + kOffSmall);
  uint32_t* s_key = reinterpret_cast<uint32_t*>(smem + kOffKeys);
  const int units_cap = a.rows_per_cta;                                 // rows (flat) or blocks (pooled)
  int* s_pool = reinterpret_cast<int*>(s_key + key_words(POOLED ? units_cap * kBlock : units_cap));

  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank(), ncta = cluster_size();

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumers);
    }
    mbar_fence_init();
    sm.failed = 0u;
  }
  pdl_wait();   // the pool / n_pool come from the preceding launch
  const int nv = clamp_count(a.n_valid[b], a.valid_cap, a.err);

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
  const uint8_t* keys = static_cast<const uint8_t*>(a.keys) + (long long)(b / a.seq_div) * a.rows_per_seq * kRowBytes;
  if (warp == kConsumers) {
    const uint64_t pol = l2_evict_first();   // every key row is read once
    int i = 0;
    for (; i < ntiles; ++i) {
      const int s = i % kStages;
      bool ok = true;
      if (lane == 0 && i >= kStages) ok = mbar_wait(&sm.empty[s], ((i / kStages) - 1) & 1, a.wait_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* dst = tiles + s * kTileBytes;
      const bool copy = !(a.skip_first_copy && i == 0);   // test hook: tile 0's barrier never completes
      if (!POOLED) {
        if (lane == 0) {
          const int r0 = begin + i * kTileRows;
          const uint32_t bytes = uint32_t(min(kTileRows, end - r0)) * kRowBytes;
          mbar_arrive_expect_tx(&sm.full[s], bytes);
          if (copy) bulk_g2s_hint(dst, keys + (long long)r0 * kRowBytes, bytes, &sm.full[s], pol);
        }
      } else {
        const int p0 = i * kBlocksPerTile;
        const int np = min(kBlocksPerTile, n_loc_units - p0);
        const int blk = lane < np ? s_pool[p0 + lane] : -1;
        const unsigned have = __ballot_sync(0xffffffffu, blk >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], uint32_t(__popc(have)) * kBlockBytes);
        __syncwarp();
        if (blk >= 0 && copy)
          bulk_g2s_hint(dst + lane * kBlockBytes, keys + (long long)blk * kBlockBytes, kBlockBytes, &sm.full[s], pol);
      }
    }
    if (lane == 0) {
      if (i < ntiles) {
        report(a.err, kErrTimeout, i);
        sm.failed = 1u;
      }
      // every copy issued has landed (or its wait gave up) before the ring is reused
      for (int j = max(0, i - kStages); j < i; ++j)
        if (!mbar_wait(&sm.full[j % kStages], (j / kStages) & 1, a.wait_ns)) sm.failed = 1u;
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
      if (!mbar_wait(&sm.full[s], (i / kStages) & 1, a.wait_ns)) {
        report(a.err, kErrTimeout, i);
        sm.failed = 1u;
        break;
      }
      const uint8_t* tile = tiles + s * kTileBytes;
      (void)tile;
      uint32_t ra[kMTiles][8], rb[kMTiles][8];
#pragma unroll
      for (int m = 0; m < kMTiles; ++m) {
        const uint8_t* p = tile + ((warp * kMTiles + m) * 16 + g) * kRowBytes + 32 * t;
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
      for (int m = 0; m < kMTiles; ++m) {
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
        const int row = i * kTileRows + (warp * kMTiles + m) * 16 + g + 8 * t;
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
  if (tid < 3 && rows_total + tid < key_words(rows_total)) s_key[rows_total + tid] = 0u;   // padding: no candidate
  __syncthreads();   // all keys written; the ring buffer is free for the histogram
  if (sm.failed) {
    // A bounded wait gave up (recorded in the error word): some keys were never
    // written.  This CTA then offers no candidate, so that the cluster's
    // selection stays consistent and every write stays in bounds.
    for (int j = tid; j < key_words(rows_total); j += kThreads) s_key[j] = 0u;
    my_cnt = 0u;
    my_lo = 0xffffffffu;
    my_hi = 0u;
    __syncthreads();
  }

  // ---------------- phase 2: cluster-wide exact Top-k over the keys
  uint32_t* ring = reinterpret_cast<uint32_t*>(smem);
  uint32_t* histD = ring;                                 // [kBins / 2][kLanes], 16-bit pairs
  uint32_t* gk = ring;                                    // gathered keys, per-CTA segments
  uint32_t* kbin = ring + kGatherWords;                   // [rows] bin of each key (bytes)
  const uint8_t* kbin8 = reinterpret_cast<const uint8_t*>(kbin);
  uint32_t* histL = ring + kGatherWords;                  // [kBins][kCopiesL], after the gather
  uint32_t* totL = histL + kBins * kCopiesL;              // [kBins]
  uint32_t* tot = ring + kRegionA;                        // [2][kMaxCluster][kBins / 2]
  const uint32_t k = uint32_t(a.k);
  const uint4* kv = reinterpret_cast<const uint4*>(s_key);   // 16-byte reads of the keys
  const int nvec = key_words(rows_total) / 4;
  if (tid == 0) sm.gcount = 0u;
  if (tid < kMaxCluster) {
    sm.above_r[tid] = 0u;
    sm.gt_g[tid] = 0u;
    sm.eq_g[tid] = 0u;
  }

  // Selected: every key > T, plus the first q keys == T in index order.
  uint32_t T = 0u, q = 0u;
  uint32_t lo = 0u, hi = 0xffffffffu, need = k;
  uint32_t fsel = 0u;            // once filtered: the members are also in bin fsel of the last pass
  bool filtered = false, gathered = false, resolved = false;
  uint32_t n_all = 0u;           // valid candidates of the query
  for (int step = 0; step < 12 && !resolved; ++step) {
    // (1) count, min and max of the members in every CTA, pushed to every CTA
    {
      uint32_t c = my_cnt, l = my_lo, h = my_hi;   // step 0: tracked while scoring
      if (step > 0) {
        c = 0u;
        l = 0xffffffffu;
        h = 0u;
        for (int j = tid; j < rows_total; j += kThreads) {
          const uint32_t kk = s_key[j];
          if (kk >= lo && kk <= hi && (!filtered || kbin8[j] == fsel)) {
            ++c;
            l = min(l, kk);
            h = max(h, kk);
          }
        }
      }
      c = __reduce_add_sync(0xffffffffu, c);
      l = __reduce_min_sync(0xffffffffu, l);
      h = __reduce_max_sync(0xffffffffu, h);
      if (lane == 0) {
        sm.red[0][warp] = c;
        sm.red[1][warp] = l;
        sm.red[2][warp] = h;
      }
      __syncthreads();
      if (tid < int(ncta)) {
        uint4 v = make_uint4(0u, 0xffffffffu, 0u, 0u);
        for (int w = 0; w < kWarpsAll; ++w) {
          v.x += sm.red[0][w];
          v.y = min(v.y, sm.red[1][w]);
          v.z = max(v.z, sm.red[2][w]);
        }
        dsmem_st_v4u(dsmem_addr(&sm.stats[crank], uint32_t(tid)), v);
      }
      cluster_arrive();
      uint4* hv = reinterpret_cast<uint4*>(histD);   // region A is written by no other CTA here
      for (int j = tid; j < kHistDWords / 4; j += kThreads) hv[j] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      cluster_wait();
    }
    uint32_t n = 0u, glo = 0xffffffffu, ghi = 0u;
    for (int r = 0; r < int(ncta); ++r) {
      const uint4 v = sm.stats[r];
      n += v.x;
      if (v.x != 0u) {
        glo = min(glo, v.y);
        ghi = max(ghi, v.z);
      }
    }
    if (step == 0) n_all = n;
    if (step == 0 && n <= k) {   // every candidate is selected
      if (tid < int(ncta)) {
        sm.gt_r[tid] = sm.stats[tid].x;
        sm.eq_r[tid] = 0u;
      }
      resolved = true;
      break;
    }
    lo = glo;   // the members are exactly the keys in [lo, hi] (bins are contiguous key ranges)
    hi = ghi;
    if (n == need) {
      T = lo - 1u;
      q = 0u;
      if (tid < int(ncta)) {
        sm.gt_r[tid] = sm.above_r[tid] + sm.stats[tid].x;
        sm.eq_r[tid] = 0u;
      }
      resolved = true;
      break;
    }
    if (lo == hi) {
      T = lo;
      q = need;
      if (tid < int(ncta)) {
        sm.gt_r[tid] = sm.above_r[tid];
        sm.eq_r[tid] = sm.stats[tid].x;
      }
      resolved = true;
      break;
    }

    // (2) radix pass over [lo, hi]: every CTA's bin totals pushed to every CTA
    const Binning bn = make_binning(lo, hi, step == 0);
    for (int i0 = tid; i0 < nvec; i0 += 2 * kThreads) {
      uint32_t kk[8], packed[2] = {0u, 0u};
      load_keys8(kv, i0, nvec, kk);
#pragma unroll
      for (int u = 0; u < 8; ++u) {   // no branch: a key outside [lo, hi] adds 0 to a clamped bin
        const uint32_t bin = min(uint32_t(kBins - 1), bin_of(kk[u], bn));
        const uint32_t inc = (kk[u] >= lo && kk[u] <= hi) ? ((bin & 1u) ? 0x10000u : 1u) : 0u;
        atomicAdd(&histD[(bin >> 1) * kLanes + (lane & (kLanes - 1))], inc);
        packed[u >> 2] |= bin << (8 * (u & 3));
      }
      kbin[i0] = packed[0];
      if (i0 + kThreads < nvec) kbin[i0 + kThreads] = packed[1];
    }
    __syncthreads();
    const int buf = step & 1;
    if (tid < kBins / 2) {   // rotated reads: conflict-free
      const uint32_t* row = histD + tid * kLanes;
      uint32_t sum = 0u;
#pragma unroll 8
      for (int c = 0; c < kLanes; ++c) sum += row[(c + tid) & (kLanes - 1)];
      uint32_t* dst = tot + buf * kTotWords + crank * (kBins / 2) + tid;   // bins 2 tid, 2 tid + 1
      for (int r = 0; r < int(ncta); ++r) dsmem_st_u32(dsmem_addr(dst, uint32_t(r)), sum);
    }
    cluster_sync_all();
    uint32_t sel, sabove;
    {
      // Every warp finds the bin (same data, same result); lane l holds bins
      // 255 - 8l - j (j = 0..7), first their totals over the CTAs.
      const uint32_t* tb = tot + buf * kTotWords;
      const int b0 = kBins - 8 - 8 * lane;
      // packed sums over the CTAs: a 16-bit half never exceeds the cluster's keys (< 65,536)
      uint4 s4 = make_uint4(0u, 0u, 0u, 0u);
      for (int r = 0; r < int(ncta); ++r) {
        const uint4 x = *reinterpret_cast<const uint4*>(tb + r * (kBins / 2) + b0 / 2);   // bins b0 .. b0 + 7
        s4.x += x.x;
        s4.y += x.y;
        s4.z += x.z;
        s4.w += x.w;
      }
      const uint32_t g[8] = {s4.w >> 16, s4.w & 0xffffu, s4.z >> 16, s4.z & 0xffffu,   // bin b0 + 7 - j
                             s4.y >> 16, s4.y & 0xffffu, s4.x >> 16, s4.x & 0xffffu};
      uint32_t local = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) local += g[j];
      uint32_t incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t before = incl - local;
      int fj = -1;
      uint32_t fabove = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (fj < 0 && before < need && before + g[j] >= need) {
          fj = j;
          fabove = before;
        }
        before += g[j];
      }
      const unsigned fm = __ballot_sync(0xffffffffu, fj >= 0);
      const int fl = fm ? __ffs(fm) - 1 : 0;
      const int sj = max(0, __shfl_sync(0xffffffffu, fj, fl));
      sabove = __shfl_sync(0xffffffffu, fabove, fl);
      sel = uint32_t(kBins - 1 - 8 * fl - sj);
      if (fm == 0u && tid == 0) report(a.err, kErrBadCount, -2);   // cannot happen: [lo, hi] holds >= need keys
      // then each CTA's keys above the chosen bin and inside it (CTA r by warp r mod 5)
      for (int r = warp; r < int(ncta); r += kWarpsAll) {
        const uint4 x = *reinterpret_cast<const uint4*>(tb + r * (kBins / 2) + b0 / 2);
        const uint32_t v[8] = {x.x & 0xffffu, x.x >> 16, x.y & 0xffffu, x.y >> 16,   // bins b0 .. b0 + 7
                               x.z & 0xffffu, x.z >> 16, x.w & 0xffffu, x.w >> 16};
        uint32_t ab = 0u, in = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t bin = uint32_t(b0 + j);
          if (bin > sel) ab += v[j];
          if (bin == sel) in += v[j];
        }
        ab = __reduce_add_sync(0xffffffffu, ab);
        in = __reduce_add_sync(0xffffffffu, in);
        if (lane == 0) {
          sm.above_r[r] += ab;
          sm.cnt_r[r] = in;
        }
      }
    }
    __syncthreads();
    need -= sabove;
    fsel = sel;
    filtered = true;
    uint32_t padded = 0u;
    for (int r = 0; r < int(ncta); ++r) padded += (sm.cnt_r[r] + 3u) & ~3u;
    if (padded <= uint32_t(kGatherWords)) {
      gathered = true;
      resolved = true;
    }
  }
  if (!resolved) report(a.err, kErrBadCount, -3);   // cannot happen: every step narrows the range

  if (gathered) {
    // (3) every CTA's keys inside the chosen bin, pushed into its segment of every CTA's gather buffer
    uint32_t my_off = 0u, G = 0u;
    for (int r = 0; r < int(ncta); ++r) {
      if (r == int(crank)) my_off = G;
      G += (sm.cnt_r[r] + 3u) & ~3u;
    }
    const uint32_t my_in = sm.cnt_r[crank];
    // members: keys in [lo, hi] whose bin byte is fsel; 16 bytes compared per read
    const uint32_t sel4 = fsel * 0x01010101u;
    const int nbv = (nvec + 3) >> 2;
    for (int v = tid; v < nbv; v += kThreads) {   // few keys match: one atomic each
      const uint4 w4 = reinterpret_cast<const uint4*>(kbin)[v];
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t m = __vcmpeq4(w[c], sel4);
        while (m != 0u) {
          const int byte = (__ffs(m) - 1) >> 3;
          m &= ~(0xffu << (8 * byte));
          const int j = 16 * v + 4 * c + byte;
          const uint32_t kk = j < rows_total ? s_key[j] : 0u;
          if (kk >= lo && kk <= hi) {
            const uint32_t p = atomicAdd(&sm.gcount, 1u);
            if (p < my_in) gk[my_off + p] = kk;
          }
        }
      }
    }
    if (tid < 3 && my_in + uint32_t(tid) < ((my_in + 3u) & ~3u)) gk[my_off + my_in + tid] = 0u;
    __syncthreads();
    {
      const int nseg = int((my_in + 3u) >> 2);   // 16-byte pieces of this CTA's segment
      for (int i = tid; i < nseg; i += kThreads) {
        const uint32_t* src = gk + my_off + 4 * i;
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        for (int r = 0; r < int(ncta); ++r)
          if (r != int(crank)) dsmem_st_v4u(dsmem_addr(src, uint32_t(r)), v);
      }
    }
    cluster_sync_all();   // the last remote access of the kernel

    // Every CTA finishes the selection alone over the G gathered words: exactly
    // the keys of the chosen bin, with zeros padding each CTA's segment to 4.
    if (G <= uint32_t(2 * kThreads)) {
      // Rank finish: the threshold T is the need-th largest gathered key, found
      // by counting for each key the keys above and equal to it.
      uint32_t x[2];
      bool have[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = tid + h * kThreads;
        x[h] = i < int(G) ? gk[i] : 0u;
        have[h] = x[h] != 0u;
      }
      if (__any_sync(0xffffffffu, have[0] || have[1])) {
        uint32_t cg[2] = {0u, 0u}, ce[2] = {0u, 0u};
        const uint4* g4 = reinterpret_cast<const uint4*>(gk);
        for (int i = 0; i < int(G >> 2); ++i) {   // the same address for every lane: a broadcast
          const uint4 v = g4[i];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              cg[h] += w[c] > x[h] ? 1u : 0u;
              ce[h] += w[c] == x[h] ? 1u : 0u;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (have[h] && cg[h] < need && need <= cg[h] + ce[h]) {   // every holder of T writes the same
            sm.sel_bin = x[h];
            sm.sel_above = need - cg[h];
          }
      }
      __syncthreads();
      T = sm.sel_bin;
      q = sm.sel_above;
      // each CTA's gathered keys above and at T
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!have[h] || x[h] < T) continue;
        const uint32_t i = uint32_t(tid + h * kThreads);
        int r = 0;
        for (uint32_t off = (sm.cnt_r[0] + 3u) & ~3u; r + 1 < int(ncta) && i >= off; off += (sm.cnt_r[r] + 3u) & ~3u)
          ++r;
        atomicAdd(x[h] > T ? &sm.gt_g[r] : &sm.eq_g[r], 1u);
      }
      __syncthreads();
      if (tid < int(ncta)) {
        sm.gt_r[tid] = sm.above_r[tid] + sm.gt_g[tid];
        sm.eq_r[tid] = sm.eq_g[tid];
      }
    } else {
      // every CTA finishes the selection alone over the G gathered words (0 = padding)
      uint4* hl = reinterpret_cast<uint4*>(histL);
      bool done = false;
      Binning lflt{};                // after the first pass: the members are also in bin lsel of lflt
      uint32_t lsel = 0u;
      bool lf = false;
      for (int it = 0; it < 12; ++it) {
        uint32_t mn = 0xffffffffu, mx = 0u, c = 0u;
        for (int i = tid; i < int(G); i += kThreads) {
          const uint32_t kk = gk[i];
          if (kk >= lo && kk <= hi && (!lf || bin_of(kk, lflt) == lsel)) {
            mn = min(mn, kk);
            mx = max(mx, kk);
            ++c;
          }
        }
        for (int j = tid; j < kBins * kCopiesL / 4; j += kThreads) hl[j] = make_uint4(0u, 0u, 0u, 0u);
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        c = __reduce_add_sync(0xffffffffu, c);
        if (lane == 0) {
          sm.red[0][warp] = c;
          sm.red[1][warp] = mn;
          sm.red[2][warp] = mx;
        }
        __syncthreads();
        c = 0u;
        mn = 0xffffffffu;
        mx = 0u;
        for (int w = 0; w < kWarpsAll; ++w) {
          c += sm.red[0][w];
          mn = min(mn, sm.red[1][w]);
          mx = max(mx, sm.red[2][w]);
        }
        lo = mn;   // the members are now exactly the keys in [lo, hi]
        hi = mx;
        if (c == need) {
          T = lo - 1u;
          q = 0u;
          done = true;
          break;
        }
        if (lo == hi) {
          T = lo;
          q = need;
          done = true;
          break;
        }
        const Binning bl = make_binning(lo, hi, it < 2);
        for (int i = tid; i < int(G); i += kThreads) {
          const uint32_t kk = gk[i];
          if (kk != 0u && kk >= lo && kk <= hi)
            atomicAdd(&histL[bin_of(kk, bl) * kCopiesL + (lane & (kCopiesL - 1))], 1u);
        }
        __syncthreads();
        for (int bin = tid; bin < kBins; bin += kThreads) {
          const uint4 x = *reinterpret_cast<const uint4*>(&histL[bin * kCopiesL]);
          const uint4 y = *reinterpret_cast<const uint4*>(&histL[bin * kCopiesL + 4]);
          totL[bin] = x.x + x.y + x.z + x.w + y.x + y.y + y.z + y.w;
        }
        __syncthreads();
        if (warp == 0) {
          uint32_t g[8], local = 0u;
  #pragma unroll
          for (int j = 0; j < 8; ++j) {
            g[j] = totL[kBins - 1 - lane * 8 - j];
            local += g[j];
          }
          uint32_t incl = local;
  #pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          uint32_t before = incl - local;
  #pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (before < need && before + g[j] >= need) {
              sm.sel_bin = uint32_t(kBins - 1 - lane * 8 - j);
              sm.sel_above = before;
            }
            before += g[j];
          }
        }
        __syncthreads();
        need -= sm.sel_above;
        lflt = bl;
        lsel = sm.sel_bin;
        lf = true;
      }
      if (!done) report(a.err, kErrBadCount, -3);   // cannot happen: every pass narrows the range
      // per CTA: gathered keys above and at the threshold
      uint32_t seg_off = 0u;
      for (int r = 0; r < int(ncta); ++r) {
        const uint32_t n = sm.cnt_r[r];
        if (r % kWarpsAll == warp) {
          uint32_t gtc = 0u, eqc = 0u;
          for (uint32_t i = lane; i < n; i += 32) {
            const uint32_t kk = gk[seg_off + i];
            gtc += kk > T ? 1u : 0u;
            eqc += kk == T ? 1u : 0u;
          }
          gtc = __reduce_add_sync(0xffffffffu, gtc);
          eqc = __reduce_add_sync(0xffffffffu, eqc);
          if (lane == 0) {
            sm.gt_r[r] = sm.above_r[r] + gtc;
            sm.eq_r[r] = q > 0u ? eqc : 0u;
          }
        }
        seg_off += (n + 3u) & ~3u;
      }
    }
  }
  __syncthreads();
  // The pooled stage lets the attention launch place its CTAs now: they fetch
  // their SWA rows while this kernel writes its ids.
  if (POOLED) pdl_launch_dependents();

  // ---------------- phase 3: this CTA's quota and offset, then its ids in ascending order
  uint32_t offset = 0u, quota = 0u;
  {
    uint32_t eqb = 0u;
    for (int r = 0; r < int(ncta); ++r) {
      const uint32_t qr = min(sm.eq_r[r], q > eqb ? q - eqb : 0u);
      if (r < int(crank)) offset += sm.gt_r[r] + qr;
      if (r == int(crank)) quota = qr;
      eqb += sm.eq_r[r];
    }
  }
  // Each warp owns a contiguous run of positions.  One pass lists, in order, the
  // positions of the run's keys above or at the threshold (flagged) in the run's
  // own stretch of a stage buffer (the ring is free now); the warps' counts give
  // every warp its first output slot, and a pass over the short lists writes the ids.
  uint32_t* stage = ring;
  const int seg = ((rows_total + kWarpsAll - 1) / kWarpsAll + 31) & ~31;
  const int p0 = warp * seg;
  const int p1 = min(rows_total, p0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  uint32_t wn = 0u, weq = 0u;
  for (int j0 = p0; j0 < p1; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t kk = j < p1 ? s_key[j] : 0u;
    const bool eq = q > 0u && kk == T;
    const bool hit = kk > T || eq;
    const unsigned mh = __ballot_sync(0xffffffffu, hit);
    if (hit) stage[p0 + wn + uint32_t(__popc(mh & lt))] = uint32_t(j) | (eq ? 0x80000000u : 0u);
    wn += uint32_t(__popc(mh));
    weq += uint32_t(__popc(__ballot_sync(0xffffffffu, eq)));
  }
  if (lane == 0) {
    sm.red[0][warp] = wn - weq;
    sm.red[1][warp] = weq;
  }
  __syncthreads();
  uint32_t gt_before = 0u, eq_before = 0u;
  for (int w = 0; w < warp; ++w) {
    gt_before += sm.red[0][w];
    eq_before += sm.red[1][w];
  }
  uint32_t slot = offset + gt_before + min(eq_before, quota);
  int* out = a.out + (long long)b * a.ld_out;
  for (uint32_t i0 = 0; i0 < wn; i0 += 32) {
    const uint32_t i = i0 + uint32_t(lane);
    const uint32_t v = i < wn ? stage[p0 + i] : 0u;
    const bool eq = i < wn && (v & 0x80000000u) != 0u;
    const unsigned me = __ballot_sync(0xffffffffu, eq);
    const bool take = i < wn && (!eq || eq_before + uint32_t(__popc(me & lt)) < quota);
    const unsigned mt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int j = int(v & 0x7fffffffu);
      int id;
      if (!POOLED)
        id = begin + j;
      else
        id = s_pool[j / kBlock] * kBlock + j % kBlock;
      out[slot + uint32_t(__popc(mt & lt))] = id;
    }
    slot += uint32_t(__popc(mt));
    eq_before += uint32_t(__popc(me));
  }
  const int selected = int(min(n_all, k));
  if (crank == 0) {
    if (a.n_out != nullptr && tid == 0) a.n_out[b] = selected;
    for (int j = selected + tid; j < a.k; j += kThreads) out[j] = -1;
  }
  // The block stage lets the next launch place its CTAs only now: with this
  // kernel's small footprint, CTAs of the pooled stage would share SMs with its
  // last clusters and slow them (measured per step: 2.5 us against a trigger
  // before the output pass).
  if (!POOLED) pdl_launch_dependents();
}

struct ClusterChoice {
  int c = 0;
  int units_per_cta = 0;
  size_t smem = 0;
};

}  // namespace

// Choose the cluster size.  A CTA's rows must fit in shared memory.  Above
// about kTargetRows rows per CTA the selection's sweeps grow long; below it its
// cluster barriers and pushes dominate (on the 128K Reindex step, batch 64, the
// 4,096 block keys of a query select fastest on 4 CTAs: 68.5 us per step against
// 70.2 on 8 and 72.1 on 2; the 16,384 pooled rows on 8).  A batch too small to
// cover the SMs takes more CTAs per query.  The choice is the largest C up to
// that target that keeps every cluster of the batch resident at once (one wave).
constexpr int kTargetRows = 1024;

static cudaError_t choose(bool pooled, int max_units, int batch, ClusterChoice& out) {
  const int unit_rows = pooled ? kBlock : 1;
  auto kern = pooled ? index_select_kernel<true> : index_select_kernel<false>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)max_units * unit_rows;
  long long target = (rows + kTargetRows - 1) / kTargetRows;
  target = max(target, (long long)((sms + batch - 1) / batch));
  // more than 8 CTAs (a non-portable cluster size) only while the whole batch's
  // clusters of that size stay in one wave at two CTAs per SM, and only when the rows alone call for that many (about kTargetRows each)
  const int cap = (batch * kMaxCluster <= 2 * sms && rows >= (long long)kMaxCluster * kTargetRows) ? kMaxCluster
                                                                                                : kPortableCluster;
  const int top = int(min(target, (long long)cap));
  ClusterChoice best;
  for (int c = max(top, 1); c >= 1; --c) {
    const int per = (max_units + c - 1) / c;
    if (c > kPortableCluster && per * unit_rows > kMaxRowsPerCta16) continue;
    if (per * unit_rows > kMaxRowsPerCta) break;
    const size_t smem = select_smem_bytes(per, pooled);
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
  return (max_units + kPortableCluster - 1) / kPortableCluster * unit_rows <= kMaxRowsPerCta;
}

cudaError_t launch_index_select(const SelectArgs& in, bool pooled, int batch, int max_units, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  // Every launch may use up to the largest shared-memory size of its mode
  // (opted in once per device); the cluster choice (an occupancy query) is
  // made once per (device, mode, size, batch) and kept in a small table
  // shared by all host threads.
  cudaError_t e = pooled ? once_per_device(kSetupSelectPooled, [] {
    cudaError_t r = cudaFuncSetAttribute(index_select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(select_smem_bytes(kMaxRowsPerCta / kBlock, true)));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(index_select_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return r;
  }) : once_per_device(kSetupSelectFlat, [] {
    cudaError_t r = cudaFuncSetAttribute(index_select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(select_smem_bytes(kMaxRowsPerCta, false)));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(index_select_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return r;
  });
  if (e != cudaSuccess) return e;
  struct Entry {
    int dev, pooled, units, batch;
    ClusterChoice ch;
  };
  static Entry cache[16];
  static int n_cache = 0;
  static std::mutex mu;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  ClusterChoice ch;
  {
    std::lock_guard<std::mutex> lock(mu);
    bool hit = false;
    for (int i = 0; i < n_cache && i < 16; ++i)
      if (cache[i].dev == dev && cache[i].pooled == int(pooled) && cache[i].units == max_units &&
          cache[i].batch == batch) {
        ch = cache[i].ch;
        hit = true;
      }
    if (!hit) {
      e = choose(pooled, max_units, batch, ch);
      if (e != cudaSuccess) return e;
      cache[n_cache % 16] = Entry{dev, int(pooled), max_units, batch, ch};
      ++n_cache;
    }
  }
  if (ch.c == 0) return cudaErrorInvalidValue;
  SelectArgs a = in;
  a.rows_per_cta = ch.units_per_cta;
  auto kern = pooled ? index_select_kernel<true> : index_select_kernel<false>;
  note_launch();
  return launch_pdl(kern, dim3(unsigned(ch.c), unsigned(batch), 1), dim3(kThreads), ch.smem, st, unsigned(ch.c), a);
}

}  // namespace csa2

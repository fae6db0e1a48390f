// Indexer scoring kernels and the block-summary-key kernel.
//
// Score of a compressed entry (or block summary key) k for one query:
//     s = sum_h w_h * ReLU(q_h . k)
// (DeepSeek V4.1 Flash architecture page, bullets "CSA2 reuse" and
// "Hierarchical indexer": 8 of the 38 CSA2 layers run an indexer; later
// decoder indexers score blocks first and then at most 16,384 candidates.)
//
// Fast path (bf16, 8 heads x 64 dims): the per-query product q_idx . K^T is a
// dense [8 x 64] x [64 x n] contraction, computed with mma.sync m16n8k16 (16
// entries x 8 heads x 16 dims per instruction).  The kernel is warp
// specialized: one producer warp streams key rows (128 B each) into a 4-stage
// shared-memory ring with bulk (TMA) copies completing on "full" mbarriers --
// one 16 KB copy per 128-row tile in flat mode, one 1 KB copy per 8-entry
// block in pooled mode, issued by 16 lanes in parallel -- and four consumer
// warps score the rows, releasing each stage on an "empty" mbarrier as soon as
// their fragments are in registers.  Each consumer thread reads the 32
// contiguous bytes of a row that its fragment needs: the dim order inside a
// k-step is permuted identically for the A (keys) and B (q_idx) fragments,
// which leaves the dot products unchanged, so no ldmatrix or swizzle is needed.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kHeads = 8;
constexpr int kDim = 64;
constexpr int kRowBytes = kDim * 2;                  // 128
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kRowBytes;    // 16 KB
constexpr int kStages = 4;
constexpr int kConsumers = 4;                        // consumer warps (2 m-tiles of 16 rows each per tile)
constexpr int kThreads = (kConsumers + 1) * 32;      // + one producer warp
constexpr int kBlock = 8;                            // entries per block (pooled fast path)
constexpr int kBlockBytes = kBlock * kRowBytes;      // 1 KB
constexpr int kBlocksPerTile = kTileRows / kBlock;   // 16
constexpr int kMaxPoolSlice = 2048;                  // pool positions per CTA held in smem

constexpr size_t kSmemTiles = size_t(kStages) * kTileBytes;
constexpr size_t kSmemBars = 2 * kStages * sizeof(uint64_t);
constexpr size_t fast_smem_bytes(bool pooled) {
  return kSmemTiles + kSmemBars + (pooled ? kMaxPoolSlice * sizeof(int) : 0);
}

template <bool POOLED>
__global__ void __launch_bounds__(kThreads) indexer_mma_kernel(const IndexerArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemTiles);
  uint64_t* empty = full + kStages;
  int* s_pool = reinterpret_cast<int*>(smem + kSmemTiles + kSmemBars);

  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();

  const int nv = clamp_count(a.n_valid[b], a.valid_cap, a.err);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    mbar_fence_init();
  }
  pdl_wait();   // the pool / n_pool come from the preceding launch

  int begin, end;
  if (!POOLED) {
    const int n = (nv + a.div - 1) / a.div;
    if (a.n_cand != nullptr && blockIdx.x == 0 && tid == 0) a.n_cand[b] = n;
    begin = blockIdx.x * a.per_cta;
    end = min(begin + a.per_cta, n);
  } else {
    const int np = clamp_count(a.n_pool[b], a.pool_cap, a.err);
    if (a.n_cand != nullptr && blockIdx.x == 0 && tid == 0) a.n_cand[b] = np * kBlock;
    begin = blockIdx.x * a.per_cta;
    end = min(begin + a.per_cta, np);
  }
  if (begin >= end) return;

  const int nb_valid = (nv + kBlock - 1) / kBlock;
  if (POOLED) {
    for (int i = tid; i < end - begin; i += kThreads) {
      int blk = a.pool[(long long)b * a.pool_cap + begin + i];
      if (blk < 0 || blk >= nb_valid) {
        report(a.err, kErrBadPool, blk);
        blk = -1;
      }
      s_pool[i] = blk;
    }
  }
  __syncthreads();

  const int rows_total = POOLED ? (end - begin) * kBlock : (end - begin);
  const int ntiles = (rows_total + kTileRows - 1) / kTileRows;
  const uint8_t* keys = static_cast<const uint8_t*>(a.keys) + (long long)(b / a.seq_div) * a.rows_per_seq * kRowBytes;

  if (warp == kConsumers) {
    // ---------------- producer warp
    const uint64_t pol = l2_evict_first();   // every key row is read once
    int i = 0;
    for (; i < ntiles; ++i) {
      const int s = i % kStages;
      bool ok = true;
      if (lane == 0 && i >= kStages) ok = mbar_wait(&empty[s], ((i / kStages) - 1) & 1);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* dst = tiles + s * kTileBytes;
      if (!POOLED) {
        if (lane == 0) {
          const int r0 = begin + i * kTileRows;
          const uint32_t bytes = uint32_t(min(kTileRows, end - r0)) * kRowBytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_g2s_hint(dst, keys + (long long)r0 * kRowBytes, bytes, &full[s], pol);
        }
      } else {
        const int p0 = i * kBlocksPerTile;
        const int np = min(kBlocksPerTile, (end - begin) - p0);
        const int blk = lane < np ? s_pool[p0 + lane] : -1;
        const unsigned have = __ballot_sync(0xffffffffu, blk >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(__popc(have)) * kBlockBytes);
        __syncwarp();
        if (blk >= 0)
          bulk_g2s_hint(dst + lane * kBlockBytes, keys + (long long)blk * kBlockBytes, kBlockBytes, &full[s], pol);
      }
    }
    if (lane == 0) {
      if (i < ntiles) report(a.err, kErrTimeout, i);
      // let every copy this CTA issued land (bounded) before its shared memory is released
      for (int j = max(0, i - kStages); j < i; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1);
    }
    return;
  }

  // ---------------- consumer warps
  const int g = lane >> 2, t = lane & 3;
  // B fragments (q_idx^T, 16 dims x 8 heads per k-step): thread (g, t) holds
  // q[head g][16t .. 16t + 16).  For k-step s its k-slots {2t, 2t+1} are dims
  // 16t + 4s + {0, 1} and {2t+8, 2t+9} are dims 16t + 4s + {2, 3}; the A
  // fragments below use the same map.
  const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q_idx) +
                                                   (((long long)b * kHeads + g) * kDim + 16 * t) * 2);
  const uint4 q0 = qp[0], q1 = qp[1];
  const uint32_t qf[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const float w0 = a.w[b * kHeads + 2 * t];
  const float w1 = a.w[b * kHeads + 2 * t + 1];
  const bool relu = a.relu != 0;
  float* scores = a.scores + (long long)b * a.ld;
  int* cand = a.cand != nullptr ? a.cand + (long long)b * a.ld : nullptr;

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kStages;
    if (!mbar_wait(&full[s], (i / kStages) & 1)) {
      report(a.err, kErrTimeout, i);
      break;
    }
    const uint8_t* tile = tiles + s * kTileBytes;
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
    if (lane == 0) mbar_arrive(&empty[s]);          // the stage may be refilled
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      // two independent accumulators (even / odd k-steps) shorten the MMA chain
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      mma_bf16(c0, ra[m][0], rb[m][0], ra[m][1], rb[m][1], qf[0], qf[1]);
      mma_bf16(c1, ra[m][2], rb[m][2], ra[m][3], rb[m][3], qf[2], qf[3]);
      mma_bf16(c0, ra[m][4], rb[m][4], ra[m][5], rb[m][5], qf[4], qf[5]);
      mma_bf16(c1, ra[m][6], rb[m][6], ra[m][7], rb[m][7], qf[6], qf[7]);
      // c0/c1 [0], [1]: row g, heads 2t, 2t+1;  [2], [3]: row g+8, same heads
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
      const int row = i * kTileRows + (warp * 2 + m) * 16 + g + 8 * t;   // local row
      if (t < 2 && row < rows_total) {
        const float r = t == 0 ? r0 : r1;
        if (!POOLED) {
          const int pos = begin + row;
          scores[pos] = r;
          if (cand != nullptr) cand[pos] = pos;
        } else {
          const int lp = row / kBlock, tt = row % kBlock;
          const int blk = s_pool[lp];
          const int e = blk * kBlock + tt;
          const int pos = (begin + lp) * kBlock + tt;
          const bool valid = blk >= 0 && e < nv;
          scores[pos] = valid ? r : -__int_as_float(0x7f800000);
          cand[pos] = valid ? e : -1;
        }
      }
    }
  }
}

// Generic path: any element type, head count and dim; one thread per candidate.
__global__ void __launch_bounds__(256) indexer_generic_kernel(const IndexerArgs a, int pooled) {
  extern __shared__ float sq[];   // [heads * dim] query, then [heads] weights
  const int b = blockIdx.y;
  pdl_launch_dependents();
  pdl_wait();
  const int hd = a.heads * a.dim;
  for (int i = threadIdx.x; i < hd; i += blockDim.x)
    sq[i] = load_elem(a.q_idx, (long long)b * hd + i, a.dtype);
  for (int i = threadIdx.x; i < a.heads; i += blockDim.x) sq[hd + i] = a.w[(long long)b * a.heads + i];
  __syncthreads();

  const int pos = blockIdx.x * blockDim.x + threadIdx.x;
  const int nv = clamp_count(a.n_valid[b], a.valid_cap, a.err);
  long long row;
  int cand_id;
  if (!pooled) {
    const int n = (nv + a.div - 1) / a.div;
    if (a.n_cand != nullptr && pos == 0) a.n_cand[b] = n;
    if (pos >= n) return;
    row = pos;
    cand_id = pos;
  } else {
    const int np = clamp_count(a.n_pool[b], a.pool_cap, a.err);
    if (a.n_cand != nullptr && pos == 0) a.n_cand[b] = np * a.block;
    if (pos >= np * a.block) return;
    const int lp = pos / a.block, tt = pos % a.block;
    const int nbv = (nv + a.block - 1) / a.block;
    const int blk = a.pool[(long long)b * a.pool_cap + lp];
    if (blk < 0 || blk >= nbv) {
      if (tt == 0) report(a.err, kErrBadPool, blk);
      cand_id = -1;
      row = 0;
    } else {
      row = (long long)blk * a.block + tt;
      cand_id = row < nv ? int(row) : -1;
    }
  }
  float s = -__int_as_float(0x7f800000);
  if (cand_id >= 0) {
    const long long base = ((long long)(b / a.seq_div) * a.rows_per_seq + row) * a.dim;
    s = 0.f;
    for (int h = 0; h < a.heads; ++h) {
      float d = 0.f;
      for (int i = 0; i < a.dim; ++i)
        d = __fmaf_rn(sq[h * a.dim + i], load_elem(a.keys, base + i, a.dtype), d);
      if (a.relu) d = fmaxf(d, 0.f);
      s = __fmaf_rn(sq[hd + h], d, s);
    }
  }
  a.scores[(long long)b * a.ld + pos] = s;
  if (a.cand != nullptr) a.cand[(long long)b * a.ld + pos] = cand_id;
}

__global__ void __launch_bounds__(256) block_keys_kernel(const BlockKeyArgs a) {
  const int b = blockIdx.y;
  pdl_launch_dependents();
  pdl_wait();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)a.nb_cap * a.dim) return;
  const int j = int(i / a.dim), d = int(i % a.dim);
  const int nv = clamp_count(a.n_valid[b], a.n_entries, a.err);
  const float v = block_key_elem(a.k_idx, (long long)(b / a.seq_div) * a.n_entries, a.dim, a.block, nv, j, d, a.dtype,
                                 a.round_to_int);
  store_elem(a.kb, ((long long)b * a.nb_cap + j) * a.dim + d, a.dtype, v);
}

std::atomic<int> g_sm_count[64];

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t launch_block_keys(const BlockKeyArgs& a, int batch, cudaStream_t st) {
  const long long n = (long long)a.nb_cap * a.dim;
  if (n == 0 || batch == 0) return cudaSuccess;
  dim3 grid(unsigned((n + 255) / 256), unsigned(batch));
  note_launch();
  return launch_pdl(block_keys_kernel, grid, dim3(256), 0, st, 1, a);
}

cudaError_t launch_indexer(const IndexerArgs& in, bool pooled, bool fast, int batch, int max_units,
                           cudaStream_t st) {
  // max_units: flat -> maximum valid rows per query; pooled -> pool capacity (blocks)
  if (batch == 0 || max_units == 0) return cudaSuccess;
  IndexerArgs a = in;
  if (!fast) {
    const int positions = pooled ? max_units * a.block : max_units;
    const size_t smem = (size_t(a.heads) * a.dim + a.heads) * sizeof(float);
    dim3 grid(unsigned((positions + 255) / 256), unsigned(batch));
    note_launch();
    return launch_pdl(indexer_generic_kernel, grid, dim3(256), smem, st, 1, a, pooled ? 1 : 0);
  }
  const size_t smem = fast_smem_bytes(pooled);
  auto kern = pooled ? indexer_mma_kernel<true> : indexer_mma_kernel<false>;
  const cudaError_t e = pooled ? once_per_device(kSetupIndexerPooled, [] {
    return cudaFuncSetAttribute(indexer_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(fast_smem_bytes(true)));
  }) : once_per_device(kSetupIndexerFlat, [] {
    return cudaFuncSetAttribute(indexer_mma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(fast_smem_bytes(false)));
  });
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (per_sm < 1) per_sm = 1;
  const int slots = device_sm_count() * per_sm;
  const int granule = pooled ? kBlocksPerTile : kTileRows;
  int ctas = slots / batch;
  if (ctas < 1) ctas = 1;
  const int max_ctas = (max_units + granule - 1) / granule;
  if (ctas > max_ctas) ctas = max_ctas;
  int per_cta = (max_units + ctas - 1) / ctas;
  if (pooled && per_cta > kMaxPoolSlice) per_cta = kMaxPoolSlice;
  a.per_cta = per_cta;
  dim3 grid(unsigned((max_units + per_cta - 1) / per_cta), unsigned(batch));
  note_launch();
  return launch_pdl(kern, grid, dim3(kThreads), smem, st, 1, a);
}

}  // namespace csa2

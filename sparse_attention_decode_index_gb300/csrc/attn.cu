// Sparse gather-attention: for every query head h
//     o_h = softmax(scale * q_h [K_main[idx]; K_swa]^T) [V_main[idx]; V_swa]
// one softmax over the selected main-KV rows plus the SWA rows
// (DeepSeek V4.1 Flash architecture page, bullet "Sparse attention": each
// query reads its Top-512 main-KV entries plus a 128-token SWA window; "CSA2
// with cross-layer reuse": every mode computes its own main Q and SWA KV).
//
// Fast path (bf16, 64 heads sharing one KV head, dk 192, dv 128): the
// 512 + 128 key slots of one query are split over a thread-block cluster of
// ceil(slots / 160) CTAs (4 for the architecture's 640 slots), sized so that two
// CTAs fit per SM and every cluster of a 64-query batch is resident in one wave.
// Each CTA gathers its 160 K rows (384 B) and V rows (256 B) into padded
// shared-memory rows with one bulk (TMA) copy per row, all completing on one
// mbarrier; invalid slots (index -1, or beyond n_swa) are zero-filled and
// masked.  Four warps each own 16 heads; their Q fragments are loaded straight
// into registers while the gather is in flight.  S = Q K^T and O = P V run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with a base-2 fp32 softmax.
// The partial (m, l, O) of every CTA is merged in fixed CTA order through
// distributed shared memory: per-head factors exp2(m_c - M) / L first, then
// 16-byte remote loads of the partial O rows.  No partial touches global
// memory and the result is deterministic.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kH = 64, kDk = 192, kDv = 128;
constexpr int kSlots = 160;                       // key slots per CTA
constexpr int kNT = kSlots / 8;                   // S n-tiles (8 keys each)
constexpr int kThreads = 128;
constexpr int kKRow = kDk * 2 + 16;               // 400 B: padded so ldmatrix rows hit distinct banks
constexpr int kVRow = kDv * 2 + 16;               // 272 B
constexpr int kORow = kDv + 4;                    // fp32 partial O row (floats), 16 B multiple
constexpr int kMaxCluster = 8;

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kSlots * kKRow;     // 64,000
constexpr int kOffM = kOffV + kSlots * kVRow;     // 107,520
constexpr int kOffL = kOffM + kH * 4;
constexpr int kOffF = kOffL + kH * 4;             // [kMaxCluster][kH] merge factors
constexpr int kOffValid = kOffF + kMaxCluster * kH * 4;
constexpr int kOffBar = kOffValid + kSlots * 4;
constexpr int kSmemBytes = kOffBar + 2 * 8;
constexpr int kHalf = kSlots / 2;                 // slots per gather barrier (80)
static_assert(kH * kORow * 4 <= kSlots * kKRow, "partial O must fit in the K region");
static_assert(kSlots % 16 == 0, "PV k-steps need 16-key groups");
static_assert(kNT % 4 == 0, "each gather half covers whole n-tile pairs");

CSA2_DEV void dsmem_ld_v4(float4& v, uint32_t addr) {
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 2) attn_mma_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  float* sM = reinterpret_cast<float*>(smem + kOffM);
  float* sL = reinterpret_cast<float*>(smem + kOffL);
  float* sF = reinterpret_cast<float*>(smem + kOffF);
  int* sValid = reinterpret_cast<int*>(smem + kOffValid);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  float* sO = reinterpret_cast<float*>(smem + kOffK);   // reused after S = QK^T

  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t crank = cluster_rank(), ncta = cluster_size();

  pdl_launch_dependents();
  if (tid == 0) {
    mbar_init(&bar[0], kThreads);
    mbar_init(&bar[1], kThreads);
    mbar_fence_init();
  }
  // --- Q A-fragments for heads 16w + g and 16w + g + 8, straight from global
  uint32_t qa[kDk / 16][4];
  {
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.q) +
                                                           ((long long)b * kH + warp * 16 + g) * (kDk * 2)) + t;
    const uint32_t* q1 = q0 + 8 * (kDk / 2);
#pragma unroll
    for (int ks = 0; ks < kDk / 16; ++ks) {
      qa[ks][0] = __ldg(q0 + ks * 8);
      qa[ks][1] = __ldg(q1 + ks * 8);
      qa[ks][2] = __ldg(q0 + ks * 8 + 4);
      qa[ks][3] = __ldg(q1 + ks * 8 + 4);
    }
  }
  pdl_wait();   // the indices come from the preceding launch
  __syncthreads();

  // --- gather: thread `tid` owns key slots tid and tid + 128 of this CTA; slots
  // [0, 80) complete on bar[0] and [80, 160) on bar[1], so the first half can be
  // scored while the second is still arriving
  uint32_t tx0 = 0u, tx1 = 0u;
  const uint8_t* ksrc[2] = {nullptr, nullptr};
  const uint8_t* vsrc[2] = {nullptr, nullptr};
  const int ns = clamp_count(a.n_swa[b], a.swa, a.err);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int ls = tid + j * kThreads;
    if (ls >= kSlots) break;
    const int slot = blockIdx.x * kSlots + ls;
    if (slot < a.topk) {
      const int e = a.idx[(long long)b * a.topk + slot];
      if (e >= a.n_entries) report(a.err, kErrBadIndex, e);
      if (e >= 0 && e < a.n_entries) {
        const long long r = (long long)b * a.n_entries + e;
        ksrc[j] = static_cast<const uint8_t*>(a.k_main) + r * (kDk * 2);
        vsrc[j] = static_cast<const uint8_t*>(a.v_main) + r * (kDv * 2);
      }
    } else if (slot < a.topk + a.swa && slot - a.topk < ns) {
      const long long r = (long long)b * a.swa + (slot - a.topk);
      ksrc[j] = static_cast<const uint8_t*>(a.k_swa) + r * (kDk * 2);
      vsrc[j] = static_cast<const uint8_t*>(a.v_swa) + r * (kDv * 2);
    }
    sValid[ls] = ksrc[j] != nullptr ? 1 : 0;
    if (ksrc[j] != nullptr) {
      if (ls < kHalf)
        tx0 += kDk * 2 + kDv * 2;
      else
        tx1 += kDk * 2 + kDv * 2;
    }
  }
  mbar_arrive_expect_tx(&bar[0], tx0);
  mbar_arrive_expect_tx(&bar[1], tx1);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int ls = tid + j * kThreads;
    if (ls >= kSlots) break;
    uint64_t* hb = &bar[ls < kHalf ? 0 : 1];
    if (ksrc[j] != nullptr) {
      bulk_g2s(sK + ls * kKRow, ksrc[j], kDk * 2, hb);
      bulk_g2s(sV + ls * kVRow, vsrc[j], kDv * 2, hb);
    } else {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int i = 0; i < kDk * 2; i += 16) *reinterpret_cast<uint4*>(sK + ls * kKRow + i) = z;
      for (int i = 0; i < kDv * 2; i += 16) *reinterpret_cast<uint4*>(sV + ls * kVRow + i) = z;
    }
  }
  __syncthreads();   // zero-filled rows and slot flags visible to every warp

  // --- S = Q K^T for heads [16w, 16w + 16) x 160 keys, one half per gather barrier
  float s[kNT][4];
#pragma unroll
  for (int j = 0; j < kNT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  const uint8_t* krow = sK + ((lane & 7) + 8 * (lane >> 4)) * kKRow + ((lane >> 3) & 1) * 16;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (!mbar_wait(&bar[half], 0)) {
      // record the stall, give the copies in flight one more bounded wait
      report(a.err, kErrTimeout, b);
      mbar_wait(&bar[half], 0);
    }
#pragma unroll
    for (int ks = 0; ks < kDk / 16; ++ks) {
#pragma unroll
      for (int jp = half * kNT / 4; jp < (half + 1) * kNT / 4; ++jp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, krow + jp * 16 * kKRow + ks * 32);
        mma_bf16(s[2 * jp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16(s[2 * jp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }
  }

  // --- softmax (base 2): rows g and g + 8 of this warp's 16 heads
  const float sl2 = a.scale * 1.4426950408889634f;
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < kNT; ++j) {
    const bool v0 = sValid[8 * j + 2 * t] != 0, v1 = sValid[8 * j + 2 * t + 1] != 0;
    s[j][0] = v0 ? s[j][0] * sl2 : -INFINITY;
    s[j][1] = v1 ? s[j][1] * sl2 : -INFINITY;
    s[j][2] = v0 ? s[j][2] * sl2 : -INFINITY;
    s[j][3] = v1 ? s[j][3] * sl2 : -INFINITY;
    m0 = fmaxf(m0, fmaxf(s[j][0], s[j][1]));
    m1 = fmaxf(m1, fmaxf(s[j][2], s[j][3]));
  }
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  const float b0s = m0 == -INFINITY ? 0.f : m0;
  const float b1s = m1 == -INFINITY ? 0.f : m1;
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int j = 0; j < kNT; ++j) {
    s[j][0] = exp2f(s[j][0] - b0s);
    s[j][1] = exp2f(s[j][1] - b0s);
    s[j][2] = exp2f(s[j][2] - b1s);
    s[j][3] = exp2f(s[j][3] - b1s);
    l0 += s[j][0] + s[j][1];
    l1 += s[j][2] + s[j][3];
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // --- O = P V (P from the S accumulators, V rows via ldmatrix.trans)
  float o[kDv / 8][4];
#pragma unroll
  for (int j = 0; j < kDv / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const uint8_t* vrow = sV + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kVRow + (lane >> 4) * 16;
#pragma unroll
  for (int kk = 0; kk < kSlots / 16; ++kk) {
    const uint32_t p0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
    const uint32_t p1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
    const uint32_t p2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
    const uint32_t p3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
    for (int dp = 0; dp < kDv / 16; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(b0, b1, b2, b3, vrow + kk * 16 * kVRow + dp * 32);
      mma_bf16(o[2 * dp], p0, p1, p2, p3, b0, b1);
      mma_bf16(o[2 * dp + 1], p0, p1, p2, p3, b2, b3);
    }
  }

  // --- partial (m, l, O) of this CTA into shared memory (O over the K region)
  __syncthreads();
  const int h0 = warp * 16 + g, h1 = h0 + 8;
#pragma unroll
  for (int j = 0; j < kDv / 8; ++j) {
    *reinterpret_cast<float2*>(sO + h0 * kORow + 8 * j + 2 * t) = make_float2(o[j][0], o[j][1]);
    *reinterpret_cast<float2*>(sO + h1 * kORow + 8 * j + 2 * t) = make_float2(o[j][2], o[j][3]);
  }
  if (t == 0) {
    sM[h0] = m0;
    sL[h0] = l0;
    sM[h1] = m1;
    sL[h1] = l1;
  }
  cluster_sync_all();

  // --- merge factors f_c[h] = exp2(m_c - M) / L for every CTA c (fixed order);
  // all remote loads are issued before any of them is used
  if (tid < kH) {
    const int h = tid;
    float mr[kMaxCluster], lr[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      if (r < int(ncta)) {
        mr[r] = dsmem_ld_f32(dsmem_addr(sM + h, r));
        lr[r] = dsmem_ld_f32(dsmem_addr(sL + h, r));
      } else {
        mr[r] = -INFINITY;
        lr[r] = 0.f;
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) M = fmaxf(M, mr[r]);
    float L = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (mr[r] != -INFINITY) L += exp2f(mr[r] - M) * lr[r];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < int(ncta)) sF[r * kH + h] = (M == -INFINITY || mr[r] == -INFINITY) ? 0.f : exp2f(mr[r] - M) / L;
    if (crank == 0 && a.lse != nullptr)
      a.lse[(long long)b * kH + h] = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
  }
  __syncthreads();

  // --- out[h, 4d..4d+4) = sum_c f_c[h] * O_c[h, 4d..4d+4); thread owns float4 slices.
  // The cluster has ncta * 128 threads and 64 * 32 slices: with ncta = 4 every
  // thread owns exactly 4 slices; all their remote loads are issued up front.
  constexpr int kSlices = kH * kDv / 4;
  const int nthreads = int(ncta) * kThreads;
  for (int e0 = int(crank) * kThreads + tid; e0 < kSlices; e0 += 4 * nthreads) {
    float4 v[4][kMaxCluster];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * nthreads;
      const int h = e / (kDv / 4), d4 = e % (kDv / 4);
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (e < kSlices && r < int(ncta)) dsmem_ld_v4(v[u][r], dsmem_addr(sO + h * kORow + 4 * d4, r));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * nthreads;
      if (e >= kSlices) break;
      const int h = e / (kDv / 4), d4 = e % (kDv / 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r >= int(ncta)) break;
        const float f = sF[r * kH + h];
        acc.x += f * v[u][r].x;
        acc.y += f * v[u][r].y;
        acc.z += f * v[u][r].z;
        acc.w += f * v[u][r].w;
      }
      *reinterpret_cast<float4*>(a.out + ((long long)b * kH + h) * kDv + 4 * d4) = acc;
    }
  }
  cluster_sync_all();
}

// Generic path: any head count / dims / element type; one CTA per (query, head).
__global__ void __launch_bounds__(128) attn_generic_kernel(const AttnArgs a) {
  extern __shared__ float sh[];
  const int b = blockIdx.y, h = blockIdx.x, tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int nslots = a.topk + a.swa;
  float* sq = sh;                       // [k_dim]
  float* sp = sh + a.k_dim;             // [nslots] logits -> probabilities
  float* red = sp + nslots;             // [32]
  for (int i = tid; i < a.k_dim; i += blockDim.x)
    sq[i] = load_elem(a.q, ((long long)b * a.heads + h) * a.k_dim + i, a.dtype);
  __syncthreads();
  const int ns = clamp_count(a.n_swa[b], a.swa, a.err);
  float mx = -INFINITY;
  for (int j = tid; j < nslots; j += blockDim.x) {
    const void* kb = nullptr;
    long long r = 0;
    if (j < a.topk) {
      const int e = a.idx[(long long)b * a.topk + j];
      if (e >= a.n_entries && h == 0) report(a.err, kErrBadIndex, e);
      if (e >= 0 && e < a.n_entries) {
        kb = a.k_main;
        r = (long long)b * a.n_entries + e;
      }
    } else if (j - a.topk < ns) {
      kb = a.k_swa;
      r = (long long)b * a.swa + (j - a.topk);
    }
    float v = -INFINITY;
    if (kb != nullptr) {
      float d = 0.f;
      for (int i = 0; i < a.k_dim; ++i) d = __fmaf_rn(sq[i], load_elem(kb, r * a.k_dim + i, a.dtype), d);
      v = d * a.scale;
    }
    sp[j] = v;
    mx = fmaxf(mx, v);
  }
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int w = 1; w < int(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
  __syncthreads();
  float sum = 0.f;
  for (int j = tid; j < nslots; j += blockDim.x) {
    const float p = mx == -INFINITY ? 0.f : expf(sp[j] - mx);
    sp[j] = p;
    sum += p;
  }
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((tid & 31) == 0) red[tid >> 5] = sum;
  __syncthreads();
  sum = 0.f;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) sum += red[w];
  for (int d = tid; d < a.v_dim; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < nslots; ++j) {
      const float p = sp[j];
      if (p == 0.f) continue;
      long long r;
      const void* vb;
      if (j < a.topk) {
        vb = a.v_main;
        r = (long long)b * a.n_entries + a.idx[(long long)b * a.topk + j];
      } else {
        vb = a.v_swa;
        r = (long long)b * a.swa + (j - a.topk);
      }
      acc = __fmaf_rn(p, load_elem(vb, r * a.v_dim + d, a.dtype), acc);
    }
    a.out[((long long)b * a.heads + h) * a.v_dim + d] = mx == -INFINITY ? 0.f : acc / sum;
  }
  if (tid == 0 && a.lse != nullptr)
    a.lse[(long long)b * a.heads + h] = mx == -INFINITY ? -INFINITY : mx + logf(sum);
}

}  // namespace

cudaError_t launch_attn(const AttnArgs& a, bool fast, int batch, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  if (!fast) {
    const size_t smem = (size_t(a.k_dim) + a.topk + a.swa + 32) * sizeof(float);
    dim3 grid(unsigned(a.heads), unsigned(batch));
    note_launch();
    return launch_pdl(attn_generic_kernel, grid, dim3(128), smem, st, 1, a);
  }
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int ncta = (a.topk + a.swa + kSlots - 1) / kSlots;
  note_launch();
  return launch_pdl(attn_mma_kernel, dim3(unsigned(ncta), unsigned(batch), 1), dim3(kThreads), kSmemBytes, st,
                    unsigned(ncta), a);
}

int attn_max_cluster() { return kMaxCluster; }
int attn_slots_per_cta() { return kSlots; }

}  // namespace csa2

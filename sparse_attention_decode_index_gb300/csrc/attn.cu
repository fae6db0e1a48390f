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
// shared-memory rows with 16-byte cp.async copies -- consecutive threads copy
// consecutive 16-byte pieces of one row, so every row is read contiguously --
// in two commit groups (slots 0..79, 80..159) so the first half of the keys
// can be scored while the second is still arriving.  (Per-row bulk copies were
// measured to be limited by the rate at which the TMA unit accepts small
// copies.)  Invalid slots (index -1, or beyond n_swa) are zero-filled by the
// copies themselves and masked.  Four warps each own 16 heads; their Q fragments are loaded straight
// into registers while the gather is in flight.  S = Q K^T and O = P V run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with a base-2 fp32 softmax.
// The partials of the cluster are merged through distributed shared memory
// with remote stores only: every CTA writes its per-head (m, l) into every
// CTA, scales its own partial O by exp2(m_c - M) / L and pushes it to the CTA
// that owns those heads, which sums the pushed partials in fixed CTA order.
// No partial touches global memory and the result is deterministic.
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
constexpr int kOffM = kOffV + kSlots * kVRow;     // 107,520: [kMaxCluster][kH] m of every CTA
constexpr int kOffL = kOffM + kMaxCluster * kH * 4;   // [kMaxCluster][kH] l of every CTA
constexpr int kOffValid = kOffL + kMaxCluster * kH * 4;
constexpr int kOffSrc = kOffValid + kSlots * 4;            // [kSlots] K row, then [kSlots] V row addresses
constexpr int kSmemBytes = kOffSrc + 2 * kSlots * 8;
constexpr int kHalf = kSlots / 2;                 // slots per gather barrier (80)
// pushed partials: [ncta][ceil(kH / ncta)][kDv] floats in the (dead) K region
static_assert((kH + kMaxCluster - 1) * kDv * 4 <= kSlots * kKRow, "pushed partials must fit in the K region");
static_assert(kSlots % 16 == 0, "PV k-steps need 16-key groups");
static_assert(kNT % 4 == 0, "each gather half covers whole n-tile pairs");

__global__ void __launch_bounds__(kThreads, 2) attn_mma_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  float* sM = reinterpret_cast<float*>(smem + kOffM);
  float* sL = reinterpret_cast<float*>(smem + kOffL);
  int* sValid = reinterpret_cast<int*>(smem + kOffValid);
  const uint8_t** sKsrc = reinterpret_cast<const uint8_t**>(smem + kOffSrc);
  const uint8_t** sVsrc = sKsrc + kSlots;
  float* sRecv = reinterpret_cast<float*>(smem + kOffK);   // pushed partials, after S and PV everywhere

  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t crank = cluster_rank(), ncta = cluster_size();

  pdl_launch_dependents();
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

  // --- source rows of this CTA's 160 key slots (null: invalid slot)
  const int ns = clamp_count(a.n_swa[b], a.swa, a.err);
  for (int ls = tid; ls < kSlots; ls += kThreads) {
    const int slot = blockIdx.x * kSlots + ls;
    const uint8_t* ks = nullptr;
    const uint8_t* vs = nullptr;
    if (slot < a.topk) {
      const int e = a.idx[(long long)b * a.topk + slot];
      if (e >= a.n_entries) report(a.err, kErrBadIndex, e);
      if (e >= 0 && e < a.n_entries) {
        const long long r = (long long)b * a.n_entries + e;
        ks = static_cast<const uint8_t*>(a.k_main) + r * (kDk * 2);
        vs = static_cast<const uint8_t*>(a.v_main) + r * (kDv * 2);
      }
    } else if (slot < a.topk + a.swa && slot - a.topk < ns) {
      const long long r = (long long)b * a.swa + (slot - a.topk);
      ks = static_cast<const uint8_t*>(a.k_swa) + r * (kDk * 2);
      vs = static_cast<const uint8_t*>(a.v_swa) + r * (kDv * 2);
    }
    sKsrc[ls] = ks;
    sVsrc[ls] = vs;
    sValid[ls] = ks != nullptr ? 1 : 0;
  }
  __syncthreads();

  // --- gather: 16-byte pieces, 24 per K row and 16 per V row; two commit groups
  constexpr int kPieces = (kDk * 2 + kDv * 2) / 16;        // 40 per slot
  const uint8_t* zsrc = static_cast<const uint8_t*>(a.k_main);   // any valid address (0 bytes read)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    for (int c = tid; c < kHalf * kPieces; c += kThreads) {
      const int ls = half * kHalf + c / kPieces, part = c % kPieces;
      const bool isk = part < (kDk * 2) / 16;
      const uint8_t* row = isk ? sKsrc[ls] : sVsrc[ls];
      const int off = isk ? part * 16 : (part - (kDk * 2) / 16) * 16;
      uint8_t* dst = isk ? sK + ls * kKRow + off : sV + ls * kVRow + off;
      const uint32_t n = row != nullptr ? 16u : 0u;          // 0 source bytes: zero fill
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                   "l"(row != nullptr ? row + off : zsrc), "r"(n)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  // --- S = Q K^T for heads [16w, 16w + 16) x 160 keys, one half per commit group
  float s[kNT][4];
#pragma unroll
  for (int j = 0; j < kNT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  const uint8_t* krow = sK + ((lane & 7) + 8 * (lane >> 4)) * kKRow + ((lane >> 3) & 1) * 16;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (half == 0)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
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

  // --- merge across the cluster (remote stores only)
  const int h0 = warp * 16 + g, h1 = h0 + 8;
  // 1. every CTA's (m, l) of every head into every CTA: table [rank][head]
  if (t == 0) {
    for (uint32_t r = 0; r < ncta; ++r) {
      dsmem_st_f32(dsmem_addr(sM + crank * kH + h0, r), m0);
      dsmem_st_f32(dsmem_addr(sL + crank * kH + h0, r), l0);
      dsmem_st_f32(dsmem_addr(sM + crank * kH + h1, r), m1);
      dsmem_st_f32(dsmem_addr(sL + crank * kH + h1, r), l1);
    }
  }
  cluster_sync_all();   // tables complete; every CTA is past its S and PV (K/V regions free)
  // 2. own factor exp2(m_own - M) / L for rows h0, h1; scale and push to the head's owner
  const int per_owner = (kH + int(ncta) - 1) / int(ncta);
  float f0 = 0.f, f1 = 0.f;
  {
    float M0 = -INFINITY, M1 = -INFINITY;
    for (uint32_t r = 0; r < ncta; ++r) {
      M0 = fmaxf(M0, sM[r * kH + h0]);
      M1 = fmaxf(M1, sM[r * kH + h1]);
    }
    float L0 = 0.f, L1 = 0.f;
    for (uint32_t r = 0; r < ncta; ++r) {
      const float a0 = sM[r * kH + h0], a1 = sM[r * kH + h1];
      if (a0 != -INFINITY) L0 += exp2f(a0 - M0) * sL[r * kH + h0];
      if (a1 != -INFINITY) L1 += exp2f(a1 - M1) * sL[r * kH + h1];
    }
    if (M0 != -INFINITY && m0 != -INFINITY) f0 = exp2f(m0 - M0) / L0;
    if (M1 != -INFINITY && m1 != -INFINITY) f1 = exp2f(m1 - M1) / L1;
  }
  {
    const uint32_t own0 = uint32_t(h0 / per_owner), own1 = uint32_t(h1 / per_owner);
    float* dst0 = sRecv + ((size_t)crank * per_owner + (h0 - int(own0) * per_owner)) * kDv;
    float* dst1 = sRecv + ((size_t)crank * per_owner + (h1 - int(own1) * per_owner)) * kDv;
#pragma unroll
    for (int j = 0; j < kDv / 8; ++j) {
      dsmem_st_v2(dsmem_addr(dst0 + 8 * j + 2 * t, own0), o[j][0] * f0, o[j][1] * f0);
      dsmem_st_v2(dsmem_addr(dst1 + 8 * j + 2 * t, own1), o[j][2] * f1, o[j][3] * f1);
    }
  }
  cluster_sync_all();   // every pushed partial has landed in its owner
  // 3. the owner sums its heads in CTA order and writes out / lse
  const int hb = int(crank) * per_owner, he = min(kH, hb + per_owner);
  for (int e = tid; e < (he - hb) * (kDv / 4); e += kThreads) {
    const int hl = e / (kDv / 4), d4 = e % (kDv / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t r = 0; r < ncta; ++r) {
      const float4 v = *reinterpret_cast<const float4*>(sRecv + ((size_t)r * per_owner + hl) * kDv + 4 * d4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<float4*>(a.out + ((long long)b * kH + hb + hl) * kDv + 4 * d4) = acc;
  }
  if (a.lse != nullptr && tid < he - hb) {
    const int h = hb + tid;
    float M = -INFINITY;
    for (uint32_t r = 0; r < ncta; ++r) M = fmaxf(M, sM[r * kH + h]);
    float L = 0.f;
    for (uint32_t r = 0; r < ncta; ++r)
      if (sM[r * kH + h] != -INFINITY) L += exp2f(sM[r * kH + h] - M) * sL[r * kH + h];
    a.lse[(long long)b * kH + h] = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
  }
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

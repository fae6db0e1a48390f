// Sparse gather-attention: for every query head h
//     o_h = softmax(scale * q_h [K_main[idx]; K_swa]^T) [V_main[idx]; V_swa]
// one softmax over the selected main-KV rows plus the SWA rows
// (DeepSeek V4.1 Flash architecture page, bullet "Sparse attention": each
// query reads its Top-512 main-KV entries plus a 128-token SWA window; "CSA2
// with cross-layer reuse": every mode computes its own main Q and SWA KV).
//
// Fast path (bf16, 64 heads sharing one KV head, dk 192, dv 128): the
// 512 + 128 key slots of one query are split over a thread-block cluster of C
// CTAs (4 for the architecture's 640 slots), sized so that two CTAs fit per SM
// and every cluster of a 64-query batch is resident in one wave.  CTA c holds
// SWA rows [c * sp, (c + 1) * sp) in its first local slots and main index slots
// [c * mp, (c + 1) * mp) after them (mp = ceil(topk / C), sp = ceil(swa / C),
// mp + sp <= 160).  The SWA rows are inputs of the launch, so every CTA starts
// fetching them before it waits for the preceding launch to finish.
// Each CTA gathers its K rows (384 B) and V rows (256 B) into padded
// shared-memory rows with 16-byte cp.async copies: a warp copies one slot at a
// time, lane l taking the fixed 16-byte pieces l and l + 32 of the slot's 640
// bytes, so every row is read contiguously.  Three commit groups (SWA rows,
// then local slots below 80, then the rest) let the first half of the keys be
// scored while the second is still arriving.  (Per-row bulk copies were
// measured to be limited by the rate at which the TMA unit accepts small
// copies.)  Invalid slots (index -1, beyond n_swa, or unused) are zero-filled
// by the copies themselves and masked.  Four warps each own 16 heads; their Q
// fragments are loaded straight into registers first thing, so that they are in
// flight with the window count and the gather.  S = Q K^T and O = P V run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with a base-2 fp32 softmax.
// The partials of the cluster are merged through distributed shared memory:
// every CTA pushes its per-head (m, l) into the table of the CTA that owns
// those heads and leaves its unscaled partial O of all heads in its own K
// region (free once its warps are done with the keys and values).  After one
// cluster barrier the owner weights the partials by exp2(m_c - M) / L and sums
// them in fixed CTA order, so the result is deterministic, reading its peers'
// partials with distributed shared-memory loads; a second, split barrier keeps
// every CTA resident until its partials have been read.  (Writing the partials
// to workspace scratch in L2 instead was measured slower at small batches and
// equal at batch 64.)
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
constexpr int kMaxCluster = 8;

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kSlots * kKRow;     // 64,000
constexpr int kOffM = kOffV + kSlots * kVRow;     // 107,520: [kMaxCluster][kH] m of every CTA
constexpr int kOffL = kOffM + kMaxCluster * kH * 4;   // [kMaxCluster][kH] l of every CTA
constexpr int kOffValid = kOffL + kMaxCluster * kH * 4;
constexpr int kSmemBytes = kOffValid + kSlots * 4;
constexpr int kHalf = kSlots / 2;                 // slots per gather barrier (80)
constexpr int kPRow = kDv + 8;                    // partial O row (fp32): padded against bank conflicts
static_assert(kH * kPRow * 4 + kMaxCluster * kH * 4 <= kSlots * kKRow, "partials and weights fit the K region");
static_assert(kSlots % 16 == 0, "PV k-steps need 16-key groups");
static_assert(kNT % 4 == 0, "each gather half covers whole n-tile pairs");

__global__ void __launch_bounds__(kThreads, 2) attn_mma_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  float* sM = reinterpret_cast<float*>(smem + kOffM);
  float* sL = reinterpret_cast<float*>(smem + kOffL);
  int* sValid = reinterpret_cast<int*>(smem + kOffValid);

  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t crank = cluster_rank(), ncta = cluster_size();

  if (!a.release_at_end) pdl_launch_dependents();
  const int mp = (a.topk + int(ncta) - 1) / int(ncta);   // main index slots of this CTA
  const int sp = (a.swa + int(ncta) - 1) / int(ncta);    // SWA rows of this CTA (local slots first)

  // Slots are copied four at a time: the 4 x 40 16-byte pieces of four
  // consecutive slots (K row: pieces 0..23, V row: 24..39 of each) are 5
  // full-warp cp.async instructions; instruction k of lane l copies piece
  // 32k + l, i.e. slot (32k + l) / 40 of the four, piece (32k + l) % 40.
  const uint8_t* zsrc = static_cast<const uint8_t*>(a.k_main);   // any valid address (0 bytes read)
  int q_slot[5], q_off[5], q_dst[5];
  bool q_k[5];
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int p = 32 * k + lane;
    const int part = p % 40;
    q_slot[k] = p / 40;
    q_k[k] = part < 24;
    q_off[k] = q_k[k] ? part * 16 : (part - 24) * 16;
    q_dst[k] = q_slot[k] * (q_k[k] ? kKRow : kVRow) + q_off[k];
  }
  // Copy slots [ls0, ls0 + 4); lane j (j < 4) supplies slot ls0 + j's K and V rows (null: zero fill).
  auto copy_quad = [&](int ls0, const uint8_t* krow, const uint8_t* vrow) {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const uint8_t* kr = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(krow), q_slot[k]));
      const uint8_t* vr = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(vrow), q_slot[k]));
      const uint8_t* r = q_k[k] ? kr : vr;
      uint8_t* d = (q_k[k] ? sK + ls0 * kKRow : sV + ls0 * kVRow) + q_dst[k];
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(d)),
                   "l"(r != nullptr ? r + q_off[k] : zsrc), "r"(r != nullptr ? 16u : 0u)
                   : "memory");
    }
  };

  // --- Q A-fragments for heads 16w + g and 16w + g + 8, straight from global; issued
  // first, so that their latency overlaps the window count's.
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

  // --- group 0: this CTA's SWA rows (inputs of this launch), before waiting on the preceding one.
  // Local slots are handled in quads [4m, 4m + 4), quad m by warp m mod 4.
  const int ns = clamp_count(a.n_swa[b], a.swa, a.err);
  for (int q0 = 4 * warp; q0 < (sp & ~3); q0 += 16) {
    const int ls = q0 + (lane & 3);
    const int r = int(crank) * sp + ls;
    const bool ok = lane < 4 && r < a.swa && r < ns;
    const long long row = (long long)b * a.swa + r;
    copy_quad(q0, ok ? static_cast<const uint8_t*>(a.k_swa) + row * (kDk * 2) : nullptr,
              ok ? static_cast<const uint8_t*>(a.v_swa) + row * (kDv * 2) : nullptr);
    if (lane < 4) sValid[ls] = ok ? 1 : 0;
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  pdl_wait();   // the indices come from the preceding launch

  // --- main index of every slot of this warp's quads 4 * warp + 16i: lane l holds
  // quad i = l / 4 (slot l % 4) in e0 and quad i = 8 + l / 4 in e1 (l < 8); -1: no main row
  auto main_index = [&](int ls) -> int {
    const int lm = ls - sp;
    if (ls >= kSlots || lm < 0 || lm >= mp || int(crank) * mp + lm >= a.topk) return -1;
    return a.idx[(long long)b * a.topk + int(crank) * mp + lm];
  };
  const int e0 = main_index(4 * warp + 16 * (lane >> 2) + (lane & 3));
  const int e1 = lane < 8 ? main_index(4 * warp + 16 * (8 + (lane >> 2)) + (lane & 3)) : -1;

  // --- groups 1 and 2: the remaining quads (main rows, the last partial SWA quad, unused slots),
  // below / from local slot 80.  Lane j < 4 of a quad resolves slot q0 + j.
  const int first = sp & ~3;
#pragma unroll 1
  for (int grp = 1; grp <= 2; ++grp) {
    const int lo = grp == 1 ? first : max(first, kHalf), hi = grp == 1 ? max(first, kHalf) : kSlots;
    for (int q0 = lo + ((4 * warp - lo) & 15); q0 < hi; q0 += 16) {
      const int ls = q0 + (lane & 3);
      const int qi = (q0 - 4 * warp) >> 4;
      const int e = __shfl_sync(0xffffffffu, qi < 8 ? e0 : e1, ((qi & 7) << 2) | (lane & 3));
      const uint8_t* kr = nullptr;
      const uint8_t* vr = nullptr;
      bool ok = false;
      if (lane < 4) {
        if (ls < sp) {
          const int r = int(crank) * sp + ls;
          ok = r < a.swa && r < ns;
          const long long row = (long long)b * a.swa + r;
          kr = static_cast<const uint8_t*>(a.k_swa) + row * (kDk * 2);
          vr = static_cast<const uint8_t*>(a.v_swa) + row * (kDv * 2);
        } else {
          if (e >= a.n_entries) report(a.err, kErrBadIndex, e);
          ok = e >= 0 && e < a.n_entries;
          const long long row = (long long)(b / a.seq_div) * a.n_entries + e;
          kr = static_cast<const uint8_t*>(a.k_main) + row * (kDk * 2);
          vr = static_cast<const uint8_t*>(a.v_main) + row * (kDv * 2);
        }
        sValid[ls] = ok ? 1 : 0;
      }
      copy_quad(q0, ok ? kr : nullptr, ok ? vr : nullptr);
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
      asm volatile("cp.async.wait_group 1;" ::: "memory");   // groups 0 and 1: local slots below 80
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

  // --- merge across the cluster: every CTA pushes the (m, l) of its rows into
  // the table of the CTA that owns those heads and leaves its unscaled partial
  // O of all heads in its own shared memory (the K region, free once every
  // warp is done with the keys and values); after one cluster barrier the
  // owner weights the partials by exp2(m_c - M) / L and sums them in fixed CTA
  // order, reading its peers' partials through distributed shared memory.  A
  // second (split) barrier keeps every CTA resident until its partials are read.
  const int h0 = warp * 16 + g, h1 = h0 + 8;
  const int per_owner = (kH + int(ncta) - 1) / int(ncta);
  if (t == 0) {
    const uint32_t own0 = uint32_t(h0 / per_owner), own1 = uint32_t(h1 / per_owner);
    dsmem_st_f32(dsmem_addr(sM + crank * kH + h0, own0), m0);
    dsmem_st_f32(dsmem_addr(sL + crank * kH + h0, own0), l0);
    dsmem_st_f32(dsmem_addr(sM + crank * kH + h1, own1), m1);
    dsmem_st_f32(dsmem_addr(sL + crank * kH + h1, own1), l1);
  }
  __syncthreads();   // every warp is done with the K and V rows
  float* sP = reinterpret_cast<float*>(sK);   // [kH][kPRow] this CTA's unscaled partial O
#pragma unroll
  for (int j = 0; j < kDv / 8; ++j) {
    *reinterpret_cast<float2*>(sP + h0 * kPRow + 8 * j + 2 * t) = make_float2(o[j][0], o[j][1]);
    *reinterpret_cast<float2*>(sP + h1 * kPRow + 8 * j + 2 * t) = make_float2(o[j][2], o[j][3]);
  }
  cluster_sync_all();   // tables and partials of every CTA are complete and visible
  // the owner's weights exp2(m_r - M) / L per (CTA, head) first, after the partials
  const int hb = int(crank) * per_owner, he = min(kH, hb + per_owner);
  float* sW = sP + kH * kPRow;   // [kMaxCluster][kH]
  for (int h = hb + tid; h < he; h += kThreads) {
    float M = -INFINITY;
    for (uint32_t r = 0; r < ncta; ++r) M = fmaxf(M, sM[r * kH + h]);
    float L = 0.f;
    for (uint32_t r = 0; r < ncta; ++r) {
      const float mr = sM[r * kH + h];
      const float wr = (M == -INFINITY || mr == -INFINITY) ? 0.f : exp2f(mr - M);
      sW[r * kH + h] = wr;
      L += wr * sL[r * kH + h];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (uint32_t r = 0; r < ncta; ++r) sW[r * kH + h] *= inv;
  }
  __syncthreads();
  // Up to kItems (head, 4 columns) items per thread, every partial load of them
  // issued before any is used (each item reads one float4 from every CTA).
  constexpr int kItems = 4;
  const int n_items = (he - hb) * (kDv / 4);
  for (int e0 = tid; e0 < n_items; e0 += kItems * kThreads) {
    float4 v[kItems][kMaxCluster];
#pragma unroll
    for (int m = 0; m < kItems; ++m) {
      const int e = e0 + m * kThreads;
      const int h = hb + e / (kDv / 4), d4 = e % (kDv / 4);
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (e < n_items && r < int(ncta)) v[m][r] = dsmem_ld_v4f(dsmem_addr(sP + h * kPRow + 4 * d4, uint32_t(r)));
    }
#pragma unroll
    for (int m = 0; m < kItems; ++m) {
      const int e = e0 + m * kThreads;
      if (e >= n_items) continue;
      const int h = hb + e / (kDv / 4), d4 = e % (kDv / 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < int(ncta)) {
          const float wr = sW[r * kH + h];
          acc.x += wr * v[m][r].x;
          acc.y += wr * v[m][r].y;
          acc.z += wr * v[m][r].z;
          acc.w += wr * v[m][r].w;
        }
      *reinterpret_cast<float4*>(a.out + ((long long)b * kH + h) * kDv + 4 * d4) = acc;
    }
  }
  cluster_arrive();   // this CTA has read its peers' partials
  if (a.lse != nullptr && tid < he - hb) {
    const int h = hb + tid;
    float M = -INFINITY;
    for (uint32_t r = 0; r < ncta; ++r) M = fmaxf(M, sM[r * kH + h]);
    float L = 0.f;
    for (uint32_t r = 0; r < ncta; ++r)
      if (sM[r * kH + h] != -INFINITY) L += exp2f(sM[r * kH + h] - M) * sL[r * kH + h];
    a.lse[(long long)b * kH + h] = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
  }
  cluster_wait();     // every peer has read this CTA's partials: its shared memory may be released
  // Before another attention launch (a Reuse or SWA layer next), its CTAs are
  // let in only now: placed early, they slowed this launch's last clusters
  // (encoder stack Full + 5 Reuse: 321 -> 293 us per group step).
  if (a.release_at_end) pdl_launch_dependents();
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
        r = (long long)(b / a.seq_div) * a.n_entries + e;
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
        r = (long long)(b / a.seq_div) * a.n_entries + a.idx[(long long)b * a.topk + j];
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
  const cudaError_t e = once_per_device(kSetupAttn, [] {
    return cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  const int ncta = attn_cluster(a.topk, a.swa);
  if (ncta == 0) return cudaErrorInvalidValue;
  note_launch();
  return launch_pdl(attn_mma_kernel, dim3(unsigned(ncta), unsigned(batch), 1), dim3(kThreads), kSmemBytes, st,
                    unsigned(ncta), a);
}

// Smallest cluster whose CTAs can each hold ceil(topk / C) main and
// ceil(swa / C) SWA slots; 0 when no cluster of at most kMaxCluster can.
int attn_cluster(int topk, int swa) {
  for (int c = (topk + swa + kSlots - 1) / kSlots; c <= kMaxCluster; ++c)
    if (c >= 1 && (topk + c - 1) / c + (swa + c - 1) / c <= kSlots) return c;
  return 0;
}

}  // namespace csa2

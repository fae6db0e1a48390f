// Device-side helpers shared by the CSA2 kernels: error reporting, the
// order-preserving score key, mbarrier / bulk-copy (TMA) wrappers, warp-level
// MMA and shared-memory matrix loads, cluster (DSMEM) primitives.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

#define CSA2_DEV __device__ __forceinline__

namespace csa2 {

CSA2_DEV void report(int* err, int bit, int detail) {
  if (err != nullptr) {
    atomicOr(err, bit);
    atomicExch(err + 1, detail);
  }
}

CSA2_DEV int clamp_count(int v, int hi, int* err) {
  if (v < 0 || v > hi) {
    report(err, kErrBadCount, v);
    v = v < 0 ? 0 : hi;
  }
  return v;
}

// Order-preserving map of a float score to uint32: a > b  <=>  key(a) > key(b).
// -0 is folded onto +0 and NaN onto -inf, so the total order used for the
// Top-K is (score descending, index ascending) on the canonical values.
CSA2_DEV uint32_t score_key(float f) {
  if (f != f) f = -__int_as_float(0x7f800000);
  if (f == 0.0f) f = 0.0f;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

CSA2_DEV float key_score(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

CSA2_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

CSA2_DEV uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier

CSA2_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

CSA2_DEV void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

CSA2_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

CSA2_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Default limit of a bounded wait: 2 s.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Wait for the given phase parity; gives up after `limit_ns` (0: the default
// 2 s) and returns false.
CSA2_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = limit_ns != 0 ? limit_ns : kWaitLimitNs;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u && global_ns() - t0 > limit) return false;
  }
}

// Bulk (TMA) copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned); completion is signalled on `bar` as transaction bytes.
CSA2_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once (streamed keys): its lines are evicted before
// anything else, so a stream larger than L2 does not push out the rest.
CSA2_DEV uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy (from l2_evict_first).
CSA2_DEV void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

CSA2_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------------ programmatic dependent launch

// Wait until the preceding kernel in the stream has completed and its memory
// is visible (no-op when the kernel was launched without the programmatic
// serialization attribute).  Must precede any access to data that kernel
// produces or consumes.
CSA2_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to be scheduled (it still waits in
// pdl_wait for this kernel to complete).
CSA2_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ MMA

// D += A * B with A 16x16 (row), B 16x8 (col), bf16 inputs, fp32 accumulators.
CSA2_DEV void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

CSA2_DEV void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

CSA2_DEV void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

CSA2_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ clusters

CSA2_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

CSA2_DEV uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

CSA2_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Split form of cluster_sync_all: local work may run between the two halves.
CSA2_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
CSA2_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Address of the same shared variable in CTA `rank` of this cluster.
CSA2_DEV uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

CSA2_DEV void dsmem_st_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

CSA2_DEV void dsmem_st_v2(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
}

CSA2_DEV void dsmem_st_u32(uint32_t addr, uint32_t x) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(x) : "memory");
}

CSA2_DEV void dsmem_st_v4u(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

CSA2_DEV void dsmem_st_v4f(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

CSA2_DEV float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

CSA2_DEV float4 dsmem_ld_v4f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ------------------------------------------------------------------ element access

CSA2_DEV float load_elem(const void* base, long long i, int dtype) {
  if (dtype == 1) return static_cast<const float*>(base)[i];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

CSA2_DEV void store_elem(void* base, long long i, int dtype, float v) {
  if (dtype == 1)
    static_cast<float*>(base)[i] = v;
  else
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

// Block summary key element (b, block j, dim d): the mean of k_idx over the
// block's valid entries (j*block .. min((j+1)*block, nv) - 1), summed in entry
// order in fp32, optionally rounded half-to-even; 0 for a block with no valid
// entry.  Shared by the from-scratch and the incremental (append) kernels so
// that both give bit-identical keys.
CSA2_DEV float block_key_elem(const void* k_idx, long long row0, int dim, int block, int nv, int j, int d,
                              int dtype, int round_to_int) {
  const int r0 = j * block;
  const int c = min(block, nv - r0);
  if (c <= 0) return 0.f;
  float s = 0.f;
  for (int r = 0; r < c; ++r) s += load_elem(k_idx, (row0 + r0 + r) * dim + d, dtype);
  float v = s / float(c);
  if (round_to_int) v = rintf(v);
  return v;
}

}  // namespace csa2

// tc_util.cuh -- PTX wrappers and operand widening shared by the tcgen05
// kernels (sm_103a): mbarriers with bounded waits, named barriers, TMEM
// allocation / loads / stores, tcgen05.mma with A in TMEM, shared-memory
// descriptors, cp.async, cluster barriers and distributed shared memory, and
// the exact int8 / 2-bit-code -> fp16 widening.
#pragma once

#include "common.cuh"

namespace bitlinear {
namespace tc {

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s bound on every wait

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity` to complete.  Returns false
// if the CTA is aborting (another role timed out) or this wait timed out.
// The first test is inlined (mbar_wait below): a call costs several times
// the test itself, and most waits in the pipelines find the phase complete.
static __device__ __noinline__ bool mbar_wait_slow(unsigned long long* bar, uint32_t parity, int* abort_flag,
                                                   int* status) {
  const unsigned long long t0 = global_timer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      if (global_timer() - t0 > kTimeoutNs) {
        atomicExch(abort_flag, 1);
        atomicExch(status, (int)BITLINEAR_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity, int* abort_flag, int* status) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, status);
}
// Bounded wait that ignores the abort flag: used to drain this thread's own
// in-flight MMAs before TMEM is freed.
static __device__ __noinline__ void mbar_drain(unsigned long long* bar, uint32_t parity, int* status) {
  const unsigned long long t0 = global_timer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 63u) == 0u && global_timer() - t0 > kTimeoutNs) {
      atomicExch(status, (int)BITLINEAR_ERR_TIMEOUT);
      return;
    }
  }
}
// Bounded wait that ignores the abort flag, for the waits that keep two roles
// in step after an abort (the partner keeps completing the phases).  On timeout
// it records BITLINEAR_ERR_TIMEOUT, raises the abort flag and returns false.
static __device__ __noinline__ bool mbar_wait_lockstep_slow(unsigned long long* bar, uint32_t parity,
                                                            int* abort_flag, int* status) {
  const unsigned long long t0 = global_timer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u && global_timer() - t0 > kTimeoutNs) {
      atomicExch(abort_flag, 1);
      atomicExch(status, (int)BITLINEAR_ERR_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_lockstep(unsigned long long* bar, uint32_t parity, int* abort_flag,
                                                   int* status) {
  return mbar_try_wait(bar, parity) || mbar_wait_lockstep_slow(bar, parity, abort_flag, status);
}
// ---------------------------------------------------------------------------
// Thread-block clusters: rank, the all-thread cluster barrier, distributed
// shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders this CTA's earlier
// shared-memory writes before the other CTAs' later reads.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's (and, through an earlier CTA barrier, its CTA's) prior writes.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t cluster_addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}
// Bounded wait whose completion also acquires what other CTAs of the cluster
// released on this barrier (their remote arrivals).
static __device__ __noinline__ bool mbar_wait_cluster(unsigned long long* bar, uint32_t parity, int* abort_flag,
                                                      int* status) {
  const unsigned long long t0 = global_timer();
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 63u) == 63u) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      if (global_timer() - t0 > kTimeoutNs) {
        atomicExch(abort_flag, 1);
        atomicExch(status, (int)BITLINEAR_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
// Named barriers (bar.arrive does not block; bar.sync waits for `count` threads).
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (TMEM) (+)= A (TMEM: lane m holds row m, column c fp16 k = 2c, 2c + 1) x B (smem)
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// This warp's 32 lanes (one row each) <- 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Arrive on an mbarrier once every cp.async this thread issued so far has
// completed (the arrival does not raise the expected count).
__device__ __forceinline__ void cp_async_arrive(unsigned long long* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 16-byte global -> shared asynchronous copy; src_bytes = 0 writes zeros and
// reads nothing.  Completion: cp_async_arrive (or cp.async.wait_all) of the
// issuing thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Arrive on an mbarrier and raise its expected transaction bytes by `bytes`.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16)
// that completes `bytes` transaction bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3fffu);          // start address
  d |= (uint64_t)1u << 16;                          // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1u << 46;                          // descriptor version (sm_100 family)
  d |= (uint64_t)2u << 61;                          // swizzle mode: 128 B
  return d;
}

// Instruction descriptor: kind::f16, A = B = fp16, D = fp32, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4)                       // D format fp32
         | (0u << 7) | (0u << 10)        // A, B format fp16
         | ((uint32_t)(n >> 3) << 17)    // N / 8
         | ((uint32_t)(m >> 4) << 24);   // M / 16
}

// Order of k inside the fp16 tiles.  Both operands list the k of every group
// of four in the order (0, 2, 1, 3); a dot product does not depend on the order
// of its terms (and these partial sums are exact integers), and this order lets
// the weight codes be widened without shifting each pair into place.

// int8 x4 (k0..k3) -> fp16x2 words (k0, k2) and (k1, k3), exactly: bias the
// bytes to b + 128, place them in the mantissa of fp16 1024 (0x6400), subtract
// 1152.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t v, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = v ^ 0x80808080u;
  lo = hsub2(prmt(u, 0x64646464u, 0x4240u), 0x64806480u);
  hi = hsub2(prmt(u, 0x64646464u, 0x4341u), 0x64806480u);
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 32-bit packed word (16 codes; k = 16w + b + 4t sits in byte b at bit 2t) ->
// 8 fp16x2 words of code - 1 in the order above.  (word >> 8b') & (3 << 2t) in
// both 16-bit halves, ORed into fp16 1024 (0x6400), is 1024 + c * 4^t; scaling
// by 4^-t and subtracting 1024 * 4^-t + 1 gives c - 1 (all steps exact).
__device__ __forceinline__ void codes_to_f16x8(uint32_t w, uint32_t out[8]) {
  const uint32_t w8 = w >> 8;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t mask = 0x00030003u << (2 * t);
    const uint32_t scale = t == 0 ? 0x3C003C00u : t == 1 ? 0x34003400u : t == 2 ? 0x2C002C00u : 0x24002400u;
    const uint32_t bias = t == 0 ? 0xE401E401u : t == 1 ? 0xDC04DC04u : t == 2 ? 0xD410D410u : 0xCC40CC40u;
    out[2 * t] = hfma2((w & mask) | 0x64006400u, scale, bias);       // bytes 0, 2: k = 4t, 4t + 2
    out[2 * t + 1] = hfma2((w8 & mask) | 0x64006400u, scale, bias);  // bytes 1, 3: k = 4t + 1, 4t + 3
  }
}

}  // namespace tc
}  // namespace bitlinear

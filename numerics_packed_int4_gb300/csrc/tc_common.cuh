// Inline-PTX wrappers for the Blackwell (sm_103a) asynchronous machinery:
// mbarriers with bounded waits, TMA tensor loads, and the tcgen05 family
// (TMEM allocation, MMA, commit, TMEM loads/stores, fences).
#pragma once

#include <cuda.h>   // CUtensorMap

#include "qg_common.cuh"

namespace qg {

QG_DEVICE uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// ---- mbarrier -------------------------------------------------------------
QG_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}
QG_DEVICE void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
QG_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}
// One arrival for the whole warp: the warp's lanes synchronise, then lane 0
// arrives (barriers fed this way are initialised with one count per warp).
QG_DEVICE void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
QG_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
QG_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(1000u) : "memory");
  return ok != 0;
}

// Bounded wait.  Gives up after 'cap' polls or when another role of the CTA
// has raised 'abort'; on giving up it raises 'abort' and records a timeout in
// the device error word, and returns false.  Never traps.
QG_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t cap, volatile int* abort,
                         unsigned int* err) {
  for (uint32_t i = 0; i < cap; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 31u && *abort) return false;
  }
  *abort = 1;
  if (err) atomicExch(err, DEV_ERR_TIMEOUT);
  return false;
}

// Bounded wait that ignores 'abort': once a role has given up, the copies and
// MMAs the CTA already issued must still land before it releases its shared
// and tensor memory.  Gives up after 'cap' polls and returns false.
QG_DEVICE bool mbar_drain(uint64_t* bar, uint32_t parity, uint32_t cap) {
  for (uint32_t i = 0; i < cap; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Warp-collective bounded wait: every lane polls, the warp leaves together
// (needed before warp-collective tcgen05.st / tcgen05.ld).
QG_DEVICE bool mbar_wait_warp(uint64_t* bar, uint32_t parity, uint32_t cap, volatile int* abort,
                              unsigned int* err) {
  for (uint32_t i = 0; i < cap; ++i) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((i & 31u) == 31u && __any_sync(0xffffffffu, *abort != 0)) return false;
  }
  if ((threadIdx.x & 31) == 0) {
    *abort = 1;
    if (err) atomicExch(err, DEV_ERR_TIMEOUT);
  }
  __syncwarp();
  return false;
}

// ---- ready counter between a scheduler thread and the MMA issuer ----------
// The MMA issuer keeps its own memory traffic to a minimum: a scheduler thread
// does the mbarrier waits for it and publishes how many k-slabs are ready.
// Every shared-memory operation of the issuing thread stalls behind the MMAs
// it has queued, so the issuer re-reads the counter only when its cached copy
// runs out.
QG_DEVICE void publish_count(unsigned int* ctr, unsigned int v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" :: "r"(smem_addr(ctr)), "r"(v) : "memory");
}
// true once *ctr > idx; 'cached' holds the last value read.  Bounded like
// mbar_wait (the cap counts reads, each at least a shared-memory latency).
QG_DEVICE bool wait_count(unsigned int* ctr, unsigned int idx, unsigned int& cached, uint32_t cap,
                          volatile int* abort, unsigned int* err) {
  if (cached > idx) return true;
  for (uint32_t i = 0; i < cap; ++i) {
    unsigned int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(ctr)) : "memory");
    cached = v;
    if (v > idx) return true;
    if ((i & 63u) == 63u && *abort) return false;
  }
  *abort = 1;
  if (err) atomicExch(err, DEV_ERR_TIMEOUT);
  return false;
}


// ---- TMA ------------------------------------------------------------------
QG_DEVICE void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
QG_DEVICE void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

// ---- tcgen05 ------------------------------------------------------------------
QG_DEVICE void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_addr(dst_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
QG_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
QG_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
QG_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes made visible to the async proxy (TMA
// stores, tensor-core operand reads) that a later barrier hands them to
QG_DEVICE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[tmem] x B[smem desc]; kind::f16 (bf16 inputs, fp32 accumulate)
QG_DEVICE void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}
// D[tmem] (+)= A[smem desc] x B[smem desc]
QG_DEVICE void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}
// arrive on an mbarrier once every tcgen05 op issued so far by this thread completes
QG_DEVICE void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_addr(bar)) : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane
QG_DEVICE void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
QG_DEVICE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

QG_DEVICE void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr) : "memory");
}
QG_DEVICE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- descriptors ---------------------------------------------------------------
// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout written by TMA (rows of 128 B, 8-row atoms of 1024 B): start address,
// leading byte offset (unused for this layout, 1), stride byte offset 1024 B
// between 8-row groups, descriptor version 1, swizzle mode 2 (128 B).
QG_DEVICE uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// ---- epilogue arithmetic --------------------------------------------------
// (a0, a1) * (b0, b1), two IEEE round-to-nearest fp32 products in one packed op
QG_DEVICE void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// two fp32 -> bf16x2 (lo in the low half), round to nearest even
QG_DEVICE uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Instruction descriptor, kind::f16 with fp16 A and B, fp32 D, both K-major.
QG_HOST_DEVICE uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major.
QG_HOST_DEVICE uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace qg

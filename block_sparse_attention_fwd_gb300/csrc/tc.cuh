// Blackwell (sm_100 family) primitives used by the tcgen05 kernels: mbarriers
// with bounded waits, TMA tensor loads, TMEM allocation, tcgen05.mma with
// shared-memory descriptors, TMEM loads/stores and the fences between them.
//
// Every wait is bounded: after the launch's limit (bl_set_wait_limit, 2 s by
// default) a wait gives up and returns false, the caller records BL status
// bit kStatusTimeout and skips the rest of its work.  Before a CTA in which a
// wait gave up frees its TMEM and exits, the roles that issue asynchronous
// work wait for it with the fixed kWaitLimitNs: the producer for the last
// load of every barrier it armed, the MMA issuer for a commit behind its last
// MMA; the storing warps always wait for their bulk groups.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bl {
namespace tc {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kStatusCorrupt = 1;
constexpr int kStatusTimeout = 2;

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps until it completes or the hint (ns) runs out, instead of re-polling
// the barrier.  Polling warps would otherwise spend shared-memory bandwidth
// that the tensor core's shared-memory operands need.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// Non-blocking tests of up to three barrier phases, issued back to back so
// that their round trips overlap (on a thread that issues MMAs, one mbarrier
// operation was measured at hundreds of cycles even on a completed phase).
// Bit i of the result is set when phase i has completed.
__device__ __forceinline__ uint32_t mbar_test3(uint32_t a0, uint32_t p0, uint32_t a1, uint32_t p1,
                                               uint32_t a2, uint32_t p2) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q0, q1, q2;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n"
      " selp.u32 %0, 1, 0, q0;\n"
      " @q1 or.b32 %0, %0, 2;\n"
      " @q2 or.b32 %0, %0, 4;\n}\n"
      : "=r"(r)
      : "r"(a0), "r"(p0), "r"(a1), "r"(p1), "r"(a2), "r"(p2)
      : "memory");
  return r;
}
// Wait for the phase with the given parity to complete; false after
// kWaitLimitNs of global time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = saddr(bar);
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_sleep(a, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}
// The bounded wait of a kernel instantiation: the fixed limit, or (WL) the
// launch's limit kept in shared memory at limit_smem.
template <bool WL>
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity,
                                           const uint64_t* limit_smem);
template <>
__device__ __forceinline__ bool wait_phase<false>(uint64_t* bar, uint32_t parity,
                                                  const uint64_t*) {
  return mbar_wait(bar, parity);
}

// Polling wait (no suspend hint) with the fixed limit, for the waits a CTA
// that gave up makes before it exits.
__device__ __forceinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity) {
  const uint32_t a = saddr(bar);
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try(a, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}
// The same with a limit set at launch (kept in shared memory, read only when
// the phase is not complete at the first look).  Limits below the suspend
// hint poll without sleeping, so a limit of 0 gives up on any phase that is
// not complete at the second look.  Kernels instantiate this wait only for
// launches under a non-default limit.
__device__ __forceinline__ bool mbar_wait_limited(uint64_t* bar, uint32_t parity,
                                                  const uint64_t* limit_smem) {
  const uint32_t a = saddr(bar);
  if (mbar_try(a, parity)) return true;
  const uint64_t limit_ns = *reinterpret_cast<const volatile uint64_t*>(limit_smem);
  const bool sleep = limit_ns >= kSuspendHintNs;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (sleep ? mbar_try_sleep(a, parity) : mbar_try(a, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}
template <>
__device__ __forceinline__ bool wait_phase<true>(uint64_t* bar, uint32_t parity,
                                                 const uint64_t* limit_smem) {
  return mbar_wait_limited(bar, parity, limit_smem);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(saddr(dst)),
      "l"(m), "r"(saddr(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int x,
                                            int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(saddr(dst)),
      "l"(m), "r"(saddr(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(saddr(dst)),
      "l"(src), "r"(bytes), "r"(saddr(bar))
      : "memory");
}

// Bulk tensor reduce-add shared -> global (fp32 add into the tensor).  The
// coordinates must be non-negative; rows past the tensor's extent are
// dropped by the TMA unit.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* m, const void* src, int x,
                                                  int y, int z, int w) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(m),
      "r"(saddr(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// Bulk tensor store shared -> global; rows past the tensor's extent are
// dropped by the TMA unit.  Coordinates must be non-negative.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* m, const void* src, int x, int y,
                                             int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::
          "l"(m),
      "r"(saddr(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk group has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's earlier generic-proxy global writes before its (or,
// after a barrier, another thread's) later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Named barrier among `count` threads (id 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (MMA/TMA).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM
// Executed by one full warp.  The allocated base address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   saddr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, 128-byte swizzle, 1024-byte aligned atoms.
//   K-major operand: rows of 128 B (64 bf16 of K), 8-row atoms; sbo = 1024,
//     lbo unused; advance along K inside the 128 B row by adding k*32 bytes.
//   MN-major operand: rows of 128 B hold 64 consecutive MN elements for one K;
//     lbo = byte distance between 64-element MN chunks, sbo = byte distance
//     between groups of 8 K rows (1024 for a dense chunk).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with bf16 A/B, fp32 accumulate, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                               // D format: f32
         | (1u << 7)                             // A format: bf16
         | (1u << 10)                            // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)        // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)        // B major-ness
         | ((uint32_t)(N >> 3) << 17)            // N / 8
         | ((uint32_t)(M >> 4) << 24);           // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T (A read from TMEM, K-major by construction).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier once every tcgen05 op this thread issued completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          saddr(bar))
      : "memory");
}

}  // namespace tc
}  // namespace bl

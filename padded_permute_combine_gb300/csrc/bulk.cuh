// Bulk copies between global and shared memory (the Tensor Memory
// Accelerator's untiled cp.async.bulk) and the mbarriers that track them.
//
// Rules every caller keeps: both addresses and the size are multiples of
// 16 bytes; a load's completion is awaited only through mbar_wait, which
// gives up after kSpinLimit polls, so no kernel can spin forever on a copy
// that never lands. The caller then flags MOE_STATUS_TIMEOUT, waits once
// more (bounded) for its outstanding load, drains its bulk stores
// (bulk_wait_all covers stores only, not loads) and stops. If the second
// wait gives up too, the load may still target the CTA's shared memory after
// the CTA exits: the launch's output and the stream are then undefined and
// the caller must treat them as failed.
#pragma once

#include <cstdint>

namespace moe {

constexpr int kSpinLimit = 1 << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// One arrival completes a phase (the expect_tx arrival of the thread that
// issues the copies).
__device__ __forceinline__ void mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
// Makes initialised barriers visible to the copy unit and the other threads.
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrives on the barrier and announces `bytes` of copies completing on it.
__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Global -> shared copy whose completion counts down the barrier's bytes.
__device__ __forceinline__ void bulk_copy_in(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// The same with an L2 cache policy (from l2_policy_*).
__device__ __forceinline__ void bulk_copy_in(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Expect `bytes` on the barrier, then copy global -> shared; completion
// arrives on the barrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  mbar_expect(bar, bytes);
  bulk_copy_in(dst, src, bytes, bar);
}

// L2 policies for bulk loads: lines kept ahead of others (data read again
// soon) or evicted first (data read once).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Polls the barrier's phase with the given parity at most kSpinLimit times.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most one committed group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's earlier shared-memory accesses (generic proxy) before
// its later bulk copies (async proxy), e.g. before a load overwrites a
// buffer that the warp has just read.
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

}  // namespace moe

// Bulk-copy (TMA) and mbarrier helpers in inline PTX for sm_103a.
//
// A row of logits is brought into shared memory with one non-tensor bulk
// copy (cp.async.bulk, global -> shared, completion counted in bytes on an
// mbarrier).  Source and destination are 16-byte aligned and the size is a
// multiple of 16 bytes (the caller checks).  No cluster multicast is used.
//
// Every wait is bounded: a waiter polls try_wait and gives up after about
// kWaitLimitNs of wall time (the %globaltimer register), so a copy that never
// lands turns into an error status instead of a hang.
#pragma once

#include <stdint.h>

namespace moe_router {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // one second

// Device status codes written to the library's status word.
enum : int { kDeviceOk = 0, kDeviceWaitTimeout = 1 };

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arm the barrier for `bytes` of transaction and start the copy.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the
// time limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// Cluster launch control (sm_100 family): a running block asks to cancel the
// launch of a block of its grid that has not started yet and, when that
// succeeds, does that block's work itself.  The 16-byte response lands in
// shared memory (16-byte aligned) and completes `bytes` on an mbarrier, like
// a bulk copy.  Once a request has failed (no block left to cancel) the block
// makes no further requests.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void clc_request(void* response, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 16;"
               ::"r"(smem_addr(bar)) : "memory");
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];" ::"r"(smem_addr(response)), "r"(smem_addr(bar)) : "memory");
}

// The x index of the block a completed request cancelled, or -1 if it
// cancelled none.
__device__ __forceinline__ int clc_cancelled_x(const void* response) {
  int x = -1, ok = 0;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %1, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, r;\n\t}"
      : "+r"(x), "=r"(ok)
      : "r"(smem_addr(response))
      : "memory");
  return ok ? x : -1;
}

}  // namespace moe_router

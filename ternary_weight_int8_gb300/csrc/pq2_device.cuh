// pq2_device.cuh — device helpers shared by the libpq2 kernels (sm_103a).
//
// Inline PTX for the asynchronous copy machinery (mbarrier, 1-D bulk copy
// global -> shared) and bounded waits.  Every wait gives up after
// kWaitLimitCycles SM clocks, so a lost arrival can never hang the GPU: the
// caller records PQ2_ERR_TIMEOUT and keeps the barrier protocol balanced.
#pragma once
#include <cstdint>

#include "pq2.h"

namespace pq2 {

constexpr int kGroup = 128;          // weights / activations per group
constexpr int kGroupCodeBytes = 32;  // code bytes per group (4 codes/byte)
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz
// Longest single suspension of a waiting thread (it resumes earlier when the
// phase completes).
constexpr uint32_t kWaitSuspendNs = 20000;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// One arrival on `bar` for the whole warp, made by the lane that elect.sync
// picks, without a branch: a warp that branches around a single lane's
// arrival diverges and reconverges, which costs more than the arrival.  The
// same release semantics as mbar_arrive.  Every lane of the warp must call it.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
      "@P mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// As warp_arrive, made only when `on` (the same in every lane) is non-zero.
__device__ __forceinline__ void warp_arrive_if(uint32_t on, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred P, Q;\n\telect.sync _|P, 0xffffffff;\n\tsetp.ne.b32 Q, %1, 0;\n\t"
      "and.pred P, P, Q;\n\t@P mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(on)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// As mbar_try_wait, but a thread that finds the phase incomplete is
// suspended until it completes or `hint_ns` nanoseconds pass.  Waiting
// warps then leave the issue slots to the warps that work; without the hint
// the suspension is short and a waiting warp keeps competing for them.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSuspendNs)) {
    if (clock64() - start > kWaitLimitCycles) return false;
  }
  return true;
}

// As mbar_wait, with its own limit in SM clocks, and giving up early once
// *abort (a shared-memory flag, may be NULL) is non-zero.
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, long long limit,
                                                const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSuspendNs)) {
    if (abort && *abort) return false;
    if (clock64() - start > limit) return false;
  }
  return true;
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem,
                                         uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier over `threads` threads (a multiple of 32) of the block.
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicExch(status, code);
}

// dp4a with the first operand read as 4 unsigned bytes, the second as 4
// signed bytes: c + sum_i a_i * b_i.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

}  // namespace pq2

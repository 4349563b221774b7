// mbarrier helpers shared by the library's .cu files: init, arrive,
// arrive with an expected transaction count, and waits bounded in clock64
// cycles (a wait that runs out returns false; the caller records the
// timeout in the library's device status word and leaves).
#pragma once

#include <cstdint>

namespace lm {

constexpr long long kWaitCycles = 2000000000LL;
constexpr long long kDrainCycles = 4 * kWaitCycles;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar),
               "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          long long limit = kWaitCycles) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}
// The same, agreed by the whole warp (every lane waits, so every lane has
// acquired the phase; the warp proceeds only if all lanes saw it complete).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          long long limit = kWaitCycles) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit));
}

// This thread's cp.async copies issued so far arrive on `bar` when they
// complete (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(
                   bar)
               : "memory");
}

}  // namespace lm

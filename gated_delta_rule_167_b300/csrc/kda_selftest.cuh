// Self-test of the device-side failure report: one thread waits on an mbarrier that nothing
// arrives on, for at most `limit_ns` of the global timer, then latches KDA_ERR_TIMEOUT in the
// status word exactly as the prefill kernel does when one of its bounded waits gives up, and
// returns. No fault, trap or unbounded loop is involved; the context stays usable.
#pragma once

#include <cstdint>

#include "kda_common.cuh"

namespace kda {
namespace selftest {

__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool try_wait_parity(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__global__ void unanswered_wait_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint64_t t0 = timer_ns();
  bool done = false;
  while (!done) {  // phase 0 never completes: nothing arrives on the barrier
    done = try_wait_parity(a, 0u);
    if (timer_ns() - t0 > limit_ns) break;
  }
  if (!done) record_status(4u /* KDA_ERR_TIMEOUT */);
}

}  // namespace selftest
}  // namespace kda

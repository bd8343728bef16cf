// Asynchronous global -> shared copies (cp.async) for the kernels' table
// preloads: every thread puts all of its copies in flight before waiting, so a
// CTA's start-up costs one memory latency instead of one per copy.
#pragma once

#include <cuda_runtime.h>

namespace pent {

// 16 bytes; both addresses 16-byte aligned
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// 8 bytes; both addresses 8-byte aligned
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(sa), "l"(gmem) : "memory");
}

// wait for every copy this thread has issued (the CTA still needs a barrier
// before reading what other threads copied)
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

}  // namespace pent

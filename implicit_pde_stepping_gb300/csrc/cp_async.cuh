// Asynchronous global -> shared copies (cp.async): table preloads and row
// staging put every copy of a thread in flight before one wait, so they cost one
// memory latency instead of one per copy; the twisted kernel's ring keeps a
// fixed number of committed groups in flight.
#pragma once

#include <cuda_runtime.h>

namespace pent {

// 16 bytes; both addresses 16-byte aligned
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// 4 bytes; both addresses 4-byte aligned
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}

// 8 bytes; both addresses 8-byte aligned
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(sa), "l"(gmem) : "memory");
}

// close the group of copies issued since the last commit
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// wait until at most NPEND committed groups are still in flight
template <int NPEND>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(NPEND) : "memory");
}

// wait for every copy this thread has issued (the CTA still needs a barrier
// before reading what other threads copied)
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

}  // namespace pent

// Tensor-memory-accelerator (TMA) tiles: host-side tensor maps and the
// device-side bulk copy with its mbarrier.
//
// A 2-D tensor map describes an interleaved [rows][batch] array (batch
// fastest); one cp.async.bulk.tensor copies a box of `box_x` systems by
// `box_y` rows into shared memory and signals an mbarrier with the byte count.
// Out-of-range parts of a box are filled with zeros by the hardware.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pent {
namespace tma {

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
// The driver's tensor-map encoder, looked up once (thread-safe static init);
// null if the driver does not provide it.
inline PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// Map of an interleaved [rows][batch] array of `elem`-byte elements, boxes of
// box_x systems x box_y rows.  False if the driver refuses it (alignment: the
// base and the row pitch batch * elem must be multiples of 16 bytes).
inline bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, size_t elem,
                      long long batch, long long rows, unsigned box_x, unsigned box_y) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) % 16) != 0 || ((size_t)batch * elem) % 16 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)batch, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)batch * elem};
  const cuuint32_t box[2] = {box_x, box_y};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of a block-interleaved array: blocks of `bs` systems, each block an
// interleaved [rows][bs] array, blocks one after another (dims: system within
// the block, row, block).  Boxes of box_x systems x box_y rows of one block.
inline bool encode_3d_blocked(CUtensorMap* map, const void* base, CUtensorMapDataType type, size_t elem,
                              long long bs, long long rows, long long nblocks, unsigned box_x,
                              unsigned box_y) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) % 16) != 0 || ((size_t)bs * elem) % 16 != 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)bs, (cuuint64_t)rows, (cuuint64_t)nblocks};
  const cuuint64_t strides[2] = {(cuuint64_t)bs * elem, (cuuint64_t)bs * rows * elem};
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// device
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier, giving up after `max_ns`
// nanoseconds of the global timer; true if the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned long long max_ns) {
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!mbar_try_wait(bar, parity)) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > max_ns) return false;
  }
  return true;
}

// Box at (x = system, y = row) of `map` into shared memory at dst (16-byte
// aligned); completion is signalled on `bar`.  x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace tma
}  // namespace pent

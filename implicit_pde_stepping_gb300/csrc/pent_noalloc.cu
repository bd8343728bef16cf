// pent_factor_solve_noalloc: the per-system factor + solve without any device
// allocation.
//
// Some callers cannot call cudaMalloc.  Examples: an application that reserved
// all of the GPU's memory for its own pool at start-up and forbids libraries
// from allocating, or a time-critical loop where cudaMalloc/cudaFree are not
// acceptable because they may synchronise the device and take unbounded time.
// pent_factor_solve needs a scratch buffer for the factor coefficients
// gamma_i and delta_i, which such a caller would have to allocate.  This entry
// point instead uses one fixed scratch array that is part of the library
// image: a file-scope static __device__ array of kNoAllocScratchBytes
// (16 MiB).  Every GPU that loads the library holds these 16 MiB until the
// process exits.
//
// The caller still passes the bands, the right-hand side and (optionally)
// info; the kernel and its results are those of pent_factor_solve.  fp32
// systems of up to 512 rows go to the partitioned kernel, which keeps every
// intermediate on chip and needs no scratch at all.
#include <mutex>

#include "pent_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

// The shared scratch.  Every call writes gamma_i and delta_i of a row before
// it reads them back, so nothing in it has to start at zero and the contents a
// previous call left behind are never used.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// the status pent_factor_solve reports for the same CUDA error
inline pent_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return PENT_OK;
  if (e == cudaErrorMemoryAllocation) return PENT_ERR_ALLOC;
  return PENT_ERR_CUDA;
}

}  // namespace

extern "C" pent_status pent_factor_solve_noalloc(const void* a, const void* b, const void* c,
                                                 const void* d, const void* e, void* rhs_inout,
                                                 int N, int batch, pent_dtype dtype, int* info,
                                                 void* stream) {
  if (!a || !b || !c || !d || !e || !rhs_inout || N < 1 || batch < 1) return PENT_ERR_INVALID_ARG;
  if (dtype != PENT_F64 && dtype != PENT_F32) return PENT_ERR_INVALID_ARG;
  const void* ptrs[6] = {a, b, c, d, e, rhs_inout};
  for (const void* q : ptrs)
    if (!aligned16(q)) return PENT_ERR_INVALID_ARG;
  // fp32 systems of up to 512 rows take the partitioned kernel, which needs no scratch
  if (dtype == PENT_F32 && pent::persys_split_chunks(N) > 0) {
    const cudaError_t err = pent::persys_split(a, b, c, d, e, rhs_inout, N, batch, 0, info,
                                               static_cast<cudaStream_t>(stream));
    return status_of(err);
  }
  if (pent::persys_work_bytes(N, batch, dtype) > kNoAllocScratchBytes) return PENT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  cudaError_t err = scratch_address(&scratch);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return status_of(err);
  }
  err = dtype == PENT_F64
            ? pent::persys_thread_df(a, b, c, d, e, rhs_inout, N, batch, 0, scratch, info,
                                     static_cast<cudaStream_t>(stream))
            : pent::persys_thread(a, b, c, d, e, rhs_inout, N, batch, 0, dtype, scratch, info,
                                  static_cast<cudaStream_t>(stream));
  return status_of(err);
}

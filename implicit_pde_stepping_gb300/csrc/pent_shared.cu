// Shared-matrix batched solve, one thread per system, native arithmetic.
//
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs": forward
// substitution L g = f and back substitution R x = g (the steps for g and x)
// over the interleaved layout, one thread per system, factor computed once
// (the Constant variant).  For a cyclic plan the same sweeps carry the
// bordered correction of eqs. (11)–(12):
//   forward   g = L^{-1} f_hat,  acc_k = sum_i w_k,i g_i = h_k^T E^{-1} f_hat
//   tail      x_t = S^{-1} (f_t - acc)                         (eq. (12))
//   backward  y = R^{-1} g,  x_hat_i = y_i - u0_i x_t0 - u1_i x_t1  (eq. (11))
// so the periodic solve costs one pass, like the non-cyclic one.
//
// g is written over f in place (the page's in-place storage) and read back by
// the backward sweep.  Loads are issued kUnroll rows at a time so that each
// thread keeps several rows in flight.
#include "pent_internal.cuh"
#include "pent_native.cuh"

namespace pent {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 8;

template <typename T, bool CYC>
__global__ void __launch_bounds__(kThreads)
    k_shared_thread(const T* __restrict__ coef, const T* __restrict__ tail, T* __restrict__ X,
                    int M, int batch) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  native_shared_column<T, CYC, kUnroll>(coef, tail, X + s, M, (size_t)batch);
}

template <typename T>
cudaError_t launch_thread(const T* coef, const T* tail, T* X, int M, int batch, int cyclic,
                          cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  if (cyclic)
    k_shared_thread<T, true><<<grid, kThreads, 0, st>>>(coef, tail, X, M, batch);
  else
    k_shared_thread<T, false><<<grid, kThreads, 0, st>>>(coef, tail, X, M, batch);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t shared_thread_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  return launch_thread<double>(p.coef64, p.tail64, X, p.M, batch, p.cyclic, st);
}

cudaError_t shared_thread_f32(const pent_plan_s& p, float* X, int batch, cudaStream_t st) {
  return launch_thread<float>(p.coef32, p.tail32, X, p.M, batch, p.cyclic, st);
}

}  // namespace pent

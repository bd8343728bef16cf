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
  T* col = X + s;
  const size_t ld = (size_t)batch;
  const T* R = coef + (size_t)kR * M;
  const T* P = coef + (size_t)kP * M;
  const T* Q = coef + (size_t)kQ * M;
  const T* W0 = coef + (size_t)kW0 * M;
  const T* W1 = coef + (size_t)kW1 * M;
  const T* G = coef + (size_t)kGam * M;
  const T* D = coef + (size_t)kDel * M;
  const T* U0 = coef + (size_t)kU0 * M;
  const T* U1 = coef + (size_t)kU1 * M;

  T g1 = T(0), g2 = T(0), acc0 = T(0), acc1 = T(0);
  for (int i0 = 0; i0 < M; i0 += kUnroll) {
    T f[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      f[u] = (i < M) ? col[(size_t)i * ld] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < M) {
        const T g = R[i] * f[u] - P[i] * g2 - Q[i] * g1;
        col[(size_t)i * ld] = g;
        if (CYC) {
          acc0 += W0[i] * g;
          acc1 += W1[i] * g;
        }
        g2 = g1;
        g1 = g;
      }
    }
  }
  T xt0 = T(0), xt1 = T(0);
  if (CYC) {
    const T t0 = col[(size_t)M * ld] - acc0;
    const T t1 = col[(size_t)(M + 1) * ld] - acc1;
    xt0 = tail[0] * t0 + tail[1] * t1;
    xt1 = tail[2] * t0 + tail[3] * t1;
    col[(size_t)M * ld] = xt0;
    col[(size_t)(M + 1) * ld] = xt1;
  }
  T y1 = T(0), y2 = T(0);
  for (int i0 = M - 1; i0 >= 0; i0 -= kUnroll) {
    T gv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      gv[u] = (i >= 0) ? col[(size_t)i * ld] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      if (i >= 0) {
        const T y = gv[u] - G[i] * y1 - D[i] * y2;
        col[(size_t)i * ld] = CYC ? (y - U0[i] * xt0 - U1[i] * xt1) : y;
        y2 = y1;
        y1 = y;
      }
    }
  }
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

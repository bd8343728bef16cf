// One system's shared-matrix solve in native arithmetic, as a device function.
//
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs": forward
// substitution L g = f and back substitution R x = g with the factor computed
// once (the Constant variant), over one column of the interleaved layout; for
// a cyclic plan the sweeps carry Navon's bordering (eqs. (11)–(12)):
//   forward   g = L^{-1} f_hat,  acc_k = sum_i w_k,i g_i = h_k^T E^{-1} f_hat
//   tail      x_t = S^{-1} (f_t - acc)                         (eq. (12))
//   backward  y = R^{-1} g,  x_hat_i = y_i - u0_i x_t0 - u1_i x_t1  (eq. (11))
// g is written over f in place and read back by the backward sweep.  Used by
// the one-thread-per-system kernel and, by one thread, for the rare systems the
// double-float kernels leave to native fp64 (all zero, subnormal or non-finite
// entries, or a scale outside their exponent window).
#pragma once

#include "pent_internal.cuh"

namespace pent {

template <typename T, bool CYC, int U = 8>
__device__ __forceinline__ void native_shared_column(const T* __restrict__ coef, const T* __restrict__ tail,
                                                     T* __restrict__ col, int M, size_t ld) {
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
  for (int i0 = 0; i0 < M; i0 += U) {
    T f[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u;
      f[u] = (i < M) ? col[(size_t)i * ld] : T(0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
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
  for (int i0 = M - 1; i0 >= 0; i0 -= U) {
    T gv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 - u;
      gv[u] = (i >= 0) ? col[(size_t)i * ld] : T(0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
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

}  // namespace pent

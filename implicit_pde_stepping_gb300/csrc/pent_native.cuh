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
// the one-thread-per-system kernels and, by one thread, for the rare systems the
// double-float kernels leave to native fp64 (all zero, subnormal or non-finite
// entries, or a scale outside their exponent window).
//
// The fused time steps of the same page, one column each, follow: Cahn–Hilliard
// (eqs. (1a), (2): the right-hand side C + k2 D2(C^3 - C) built inside the
// forward sweep from C_{i-1..i+1}, which pass through the same thread) and
// Crank–Nicolson (eqs. (5)–(6): the explicit half taken as 2I - A with the
// plan's own bands).  In-place safety: the forward sweep writes g_i over C_i
// only after every later row it needs has been read, and the border rows are
// overwritten last.
#pragma once

#include "pent_internal.cuh"

namespace pent {

// a plan's native fp64 tables, for kernels that fall back to them per system
struct NativeTabs {
  const double* coef64;
  const double* tail64;
  const double* bands;
};

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

__device__ __forceinline__ double native_cubic_minus(double c) { return c * c * c - c; }

// One Cahn–Hilliard step of one column (stride ld), in place.
template <int kUnroll = 8>
__device__ __forceinline__ void native_ch_column(const double* __restrict__ coef, const double* __restrict__ tail,
                                                 double* __restrict__ col, int N, size_t ld, double k2) {
  const int M = N - 2;
  const double* R = coef + (size_t)kR * M;
  const double* P = coef + (size_t)kP * M;
  const double* Q = coef + (size_t)kQ * M;
  const double* W0 = coef + (size_t)kW0 * M;
  const double* W1 = coef + (size_t)kW1 * M;
  const double* G = coef + (size_t)kGam * M;
  const double* D = coef + (size_t)kDel * M;
  const double* U0 = coef + (size_t)kU0 * M;
  const double* U1 = coef + (size_t)kU1 * M;

  const double cLast = col[(size_t)(N - 1) * ld];
  const double c0 = col[0];
  const double uLast = native_cubic_minus(cLast);
  const double u0 = native_cubic_minus(c0);
  double uprev = uLast, ucur = u0, ccur = c0;
  double g1 = 0.0, g2 = 0.0, acc0 = 0.0, acc1 = 0.0;
  for (int i0 = 0; i0 < M; i0 += kUnroll) {
    double cn[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u + 1;   // C_{i+1} for row i0+u; row M = N-2 is still C
      cn[u] = (i <= M) ? col[(size_t)i * ld] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < M) {
        const double unext = native_cubic_minus(cn[u]);
        const double rhs = ccur + k2 * (uprev - 2.0 * ucur + unext);
        const double g = R[i] * rhs - P[i] * g2 - Q[i] * g1;
        col[(size_t)i * ld] = g;
        acc0 += W0[i] * g;
        acc1 += W1[i] * g;
        g2 = g1; g1 = g;
        uprev = ucur; ucur = unext; ccur = cn[u];
      }
    }
  }
  // now ccur = C_{N-2}, ucur = u_{N-2}, uprev = u_{N-3}
  const double f0 = ccur + k2 * (uprev - 2.0 * ucur + uLast);
  const double f1 = cLast + k2 * (ucur - 2.0 * uLast + u0);
  const double t0 = f0 - acc0, t1 = f1 - acc1;
  const double xt0 = tail[0] * t0 + tail[1] * t1;
  const double xt1 = tail[2] * t0 + tail[3] * t1;
  col[(size_t)M * ld] = xt0;
  col[(size_t)(M + 1) * ld] = xt1;
  double y1 = 0.0, y2 = 0.0;
  for (int i0 = M - 1; i0 >= 0; i0 -= kUnroll) {
    double gv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      gv[u] = (i >= 0) ? col[(size_t)i * ld] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      if (i >= 0) {
        const double y = gv[u] - G[i] * y1 - D[i] * y2;
        col[(size_t)i * ld] = y - U0[i] * xt0 - U1[i] * xt1;
        y2 = y1; y1 = y;
      }
    }
  }
}

// One Crank–Nicolson step of one column (stride ld), in place; `bands` are the
// plan's bands [5][N] of A (explicit half 2I - A).
template <int kUnroll = 8>
__device__ __forceinline__ void native_cn_column(const double* __restrict__ coef, const double* __restrict__ tail,
                                                 const double* __restrict__ bands, double* __restrict__ col, int N,
                                                 size_t ld) {
  const int M = N - 2;
  const double* R = coef + (size_t)kR * M;
  const double* P = coef + (size_t)kP * M;
  const double* Q = coef + (size_t)kQ * M;
  const double* W0 = coef + (size_t)kW0 * M;
  const double* W1 = coef + (size_t)kW1 * M;
  const double* G = coef + (size_t)kGam * M;
  const double* D = coef + (size_t)kDel * M;
  const double* U0 = coef + (size_t)kU0 * M;
  const double* U1 = coef + (size_t)kU1 * M;
  const double* Ba = bands;
  const double* Bb = bands + N;
  const double* Bc = bands + 2 * (size_t)N;
  const double* Bd = bands + 3 * (size_t)N;
  const double* Be = bands + 4 * (size_t)N;

  const double c0 = col[0], c1 = col[ld];
  const double cM = col[(size_t)M * ld], cL = col[(size_t)(M + 1) * ld];
  // window w0..w3 = C_{i-2}, C_{i-1}, C_i, C_{i+1}
  double w0 = cM, w1 = cL, w2 = c0, w3 = c1;
  double g1 = 0.0, g2 = 0.0, acc0 = 0.0, acc1 = 0.0;
  for (int i0 = 0; i0 < M; i0 += kUnroll) {
    double cn[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u + 2;   // C_{i+2} for row i0+u; rows M, M+1 are still C
      cn[u] = (i <= M + 1) ? col[(size_t)i * ld] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < M) {
        const double w4 = cn[u];
        const double ac = Ba[i] * w0 + Bb[i] * w1 + Bc[i] * w2 + Bd[i] * w3 + Be[i] * w4;
        const double rhs = 2.0 * w2 - ac;
        const double g = R[i] * rhs - P[i] * g2 - Q[i] * g1;
        col[(size_t)i * ld] = g;
        acc0 += W0[i] * g;
        acc1 += W1[i] * g;
        g2 = g1; g1 = g;
        w0 = w1; w1 = w2; w2 = w3; w3 = w4;
      }
    }
  }
  // now w0..w3 = C_{M-2}, C_{M-1}, C_M, C_{M+1}
  const double f0 = 2.0 * w2 - (Ba[M] * w0 + Bb[M] * w1 + Bc[M] * w2 + Bd[M] * w3 + Be[M] * c0);
  const double f1 =
      2.0 * w3 - (Ba[M + 1] * w1 + Bb[M + 1] * w2 + Bc[M + 1] * w3 + Bd[M + 1] * c0 + Be[M + 1] * c1);
  const double t0 = f0 - acc0, t1 = f1 - acc1;
  const double xt0 = tail[0] * t0 + tail[1] * t1;
  const double xt1 = tail[2] * t0 + tail[3] * t1;
  col[(size_t)M * ld] = xt0;
  col[(size_t)(M + 1) * ld] = xt1;
  double y1 = 0.0, y2 = 0.0;
  for (int i0 = M - 1; i0 >= 0; i0 -= kUnroll) {
    double gv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      gv[u] = (i >= 0) ? col[(size_t)i * ld] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      if (i >= 0) {
        const double y = gv[u] - G[i] * y1 - D[i] * y2;
        col[(size_t)i * ld] = y - U0[i] * xt0 - U1[i] * xt1;
        y2 = y1; y1 = y;
      }
    }
  }
}

// Out-of-line entry points for kernels that take the native path only for rare
// systems: a call keeps the native sweeps' registers out of the hot code.
__device__ __noinline__ inline void native_solve_col(const NativeTabs nt, double* col, int M, size_t ld, int cyclic) {
  if (cyclic) native_shared_column<double, true>(nt.coef64, nt.tail64, col, M, ld);
  else native_shared_column<double, false>(nt.coef64, nt.tail64, col, M, ld);
}
__device__ __noinline__ inline void native_ch_col(const NativeTabs nt, double* col, int N, size_t ld, double k2,
                                                  int nsteps) {
  for (int n = 0; n < nsteps; ++n) native_ch_column(nt.coef64, nt.tail64, col, N, ld, k2);
}
__device__ __noinline__ inline void native_cn_col(const NativeTabs nt, double* col, int N, size_t ld, int nsteps) {
  for (int n = 0; n < nsteps; ++n) native_cn_column(nt.coef64, nt.tail64, nt.bands, col, N, ld);
}
__device__ __noinline__ inline void native_hyper_col(const NativeTabs nt, double* col, int M, size_t ld, int nsteps) {
  for (int n = 0; n < nsteps; ++n) native_shared_column<double, true>(nt.coef64, nt.tail64, col, M, ld);
}

}  // namespace pent

// Fused time steps, one thread per system: explicit right-hand side + cyclic solve.
//
// Cahn–Hilliard (k_ch_thread_f64):
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs", eqs. (1a)
// and (2) with mobility D = 1, periodic on N points:
//   (I + gamma dt D4) C^{n+1} = C^n + dt D2[(C^n)^3 - C^n],  D2 = [1, -2, 1]/dx^2.
// The page builds the right-hand side with a separate stencil library before
// the solve.  Here the thread that solves system s computes its right-hand
// side on the fly inside the forward sweep: row i needs C_{i-1}, C_i, C_{i+1},
// all of which pass through the same thread, so the right-hand side never
// goes to memory.  The solve is the bordered cyclic sweep of pent_shared.cu.
//
// In-place safety: the forward sweep writes g_i over C_i only after C_{i+1}
// has been read, and rows N-2, N-1 (the border) are not overwritten until the
// end, so every C value is read before it is replaced.  C_{N-1} and C_0 are
// kept in registers for the periodic wrap.
//
// Crank–Nicolson (k_cn_thread_f64), eqs. (5)–(6) of the same page: with the
// plan's matrix A = I + sigma_x D4 (sigma_x = dt / (2 dx^4)) the explicit half
// I - sigma_x D4 equals 2I - A, so the right-hand side of row i is
//   2 C_i - (a_i C_{i-2} + b_i C_{i-1} + c_i C_i + d_i C_{i+1} + e_i C_{i+2})
// with the plan's own bands and periodic indices.  Any cyclic plan A = I + (dt/2) L
// gets its Crank–Nicolson step this way.  Row i reads C up to i+2 ahead and
// keeps C_{i-2}, C_{i-1} in registers; C_0, C_1, C_{N-2}, C_{N-1} are kept
// for the wrap.
#include "pent_internal.cuh"

namespace pent {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 8;

__device__ __forceinline__ double cubic_minus(double c) { return c * c * c - c; }

__global__ void __launch_bounds__(kThreads)
    k_ch_thread_f64(const double* __restrict__ coef, const double* __restrict__ tail,
                    double* __restrict__ X, int N, int batch, double k2) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const int M = N - 2;
  double* col = X + s;
  const size_t ld = (size_t)batch;
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
  const double uLast = cubic_minus(cLast);
  const double u0 = cubic_minus(c0);
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
        const double unext = cubic_minus(cn[u]);
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

__global__ void __launch_bounds__(kThreads)
    k_cn_thread_f64(const double* __restrict__ coef, const double* __restrict__ tail,
                    const double* __restrict__ bands, double* __restrict__ X, int N, int batch) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const int M = N - 2;
  double* col = X + s;
  const size_t ld = (size_t)batch;
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

}  // namespace

cudaError_t ch_thread_f64(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  k_ch_thread_f64<<<grid, kThreads, 0, st>>>(p.coef64, p.tail64, X, p.N, batch, k2);
  note_launch();
  return cudaGetLastError();
}

cudaError_t cn_thread_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  k_cn_thread_f64<<<grid, kThreads, 0, st>>>(p.coef64, p.tail64, p.bands, X, p.N, batch);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pent

// Device helpers shared by the plan-time factor kernels (one thread, fp64).
//
// LR factorisation of "cuPentBatch – A batched pentadiagonal solver for NVIDIA
// GPUs" (factorisation steps 1–14) over the leading M x M block of a banded
// matrix, optionally of its reversal (row i <-> M-1-i, bands a <-> e, b <-> d).
#pragma once

#include <cmath>

#include "pent_internal.cuh"

namespace pent {
namespace lr {

// band k (0..4 = a..e) of row j of the M x M leading block (or of its reversal);
// entries whose column leaves 0..M-1 are zero
__device__ inline double band(const double* bands, int N, int M, int k, int j, bool rev) {
  const int col = j + k - 2;
  if (col < 0 || col >= M) return 0.0;
  if (!rev) return bands[(size_t)k * N + j];
  return bands[(size_t)(4 - k) * N + (M - 1 - j)];
}

// rows 0..R-1: alpha, beta, gamma, delta, eps (= a).  false on a zero pivot.
__device__ inline bool factor_rows(const double* bands, int N, int M, int R, bool rev, double* al,
                                   double* be, double* ga, double* de, double* ep) {
  // blocks of 8 rows whose bands are loaded before they are used, so the
  // thread waits for memory once per block
  constexpr int kPre = 8;
  double gm1 = 0.0, gm2 = 0.0, dm1 = 0.0, dm2 = 0.0;
  for (int j0 = 0; j0 < R; j0 += kPre) {
    double bv[5][kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u)
#pragma unroll
      for (int k = 0; k < 5; ++k) bv[k][u] = (j0 + u < R) ? band(bands, N, M, k, j0 + u, rev) : 0.0;
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int j = j0 + u;
      if (j >= R) break;
      const double a = bv[0][u], b = bv[1][u], c = bv[2][u], d = bv[3][u], e = bv[4][u];
      const double beta = b - a * gm2;                 // step 8.1
      const double alpha = c - a * dm2 - beta * gm1;   // step 8.2
      if (!(alpha != 0.0) || !isfinite(alpha)) return false;
      const double ra = 1.0 / alpha;                   // one division per row
      const double g = (d - beta * dm1) * ra;          // step 8.3
      const double dd = e * ra;                        // step 8.4
      al[j] = alpha; be[j] = beta; ga[j] = g; de[j] = dd; ep[j] = a;
      gm2 = gm1; gm1 = g;
      dm2 = dm1; dm1 = dd;
    }
  }
  return true;
}

// (hi, lo) float pair of a double
__device__ inline float2 split(double v) {
  const float hi = __double2float_rn(v);
  return make_float2(hi, __double2float_rn(v - (double)hi));
}

// Border of a cyclic matrix A = [[E, G], [H^T, B]] (Navon's bordering, eq. (8)),
// E the leading M = N-2 block: columns g0, g1 of G, rows h0, h1 of H^T (all
// length M, zeroed first) and the 2x2 block B.
__device__ inline void border(const double* bands, int N, double* g0, double* g1, double* h0,
                              double* h1, double Bm[2][2]) {
  const int M = N - 2;
  const double* A = bands;
  const double* B = bands + N;
  const double* C = bands + 2 * (size_t)N;
  const double* D = bands + 3 * (size_t)N;
  const double* E = bands + 4 * (size_t)N;
  for (int i = 0; i < M; ++i) g0[i] = g1[i] = h0[i] = h1[i] = 0.0;
  g0[0] += A[0]; g1[0] += B[0]; g1[1] += A[1];
  g0[M - 2] += E[M - 2]; g0[M - 1] += D[M - 1]; g1[M - 1] += E[M - 1];
  h0[N - 4] += A[N - 2]; h0[N - 3] += B[N - 2]; h0[0] += E[N - 2];
  h1[N - 3] += A[N - 1]; h1[0] += D[N - 1]; h1[1] += E[N - 1];
  Bm[0][0] = C[N - 2]; Bm[0][1] = D[N - 2]; Bm[1][0] = B[N - 1]; Bm[1][1] = C[N - 1];
}

}  // namespace lr
}  // namespace pent

// Factorisation of a shared matrix and the precomputation of the periodic border.
//
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs":
//   - LR factorisation, factorisation steps 1–14 (done once per plan: the
//     page's split of factorisation from solve);
//   - Navon's bordering of the cyclic matrix (7c), eqs. (8)–(12): the page
//     stores the 2x2 inverse of eq. (12) and h^T E^{-1} once at start-up.
//
// The work is O(N) and serial, done once per plan, so one thread runs it.  The
// sweeps go in blocks of kPre rows whose inputs are loaded before the block is
// computed, so the thread waits for memory once per block, not once per row.
#include <cmath>

#include "pent_internal.cuh"

namespace pent {
namespace {

constexpr int kPre = 8;

__global__ void k_factor_shared(const double* __restrict__ bands, int N, int cyclic,
                                double* __restrict__ coef, double* __restrict__ tail,
                                double* __restrict__ work, int* __restrict__ status) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const int M = cyclic ? N - 2 : N;
  const double* A = bands;
  const double* B = bands + N;
  const double* C = bands + 2 * (size_t)N;
  const double* D = bands + 3 * (size_t)N;
  const double* E = bands + 4 * (size_t)N;
  double* r = coef + (size_t)kR * M;
  double* p = coef + (size_t)kP * M;
  double* q = coef + (size_t)kQ * M;
  double* w0 = coef + (size_t)kW0 * M;
  double* w1 = coef + (size_t)kW1 * M;
  double* gam = coef + (size_t)kGam * M;
  double* del = coef + (size_t)kDel * M;
  double* u0 = coef + (size_t)kU0 * M;
  double* u1 = coef + (size_t)kU1 * M;
  *status = 0;

  // Leading M x M block (the whole matrix when non-cyclic): entries whose
  // column leaves 0..M-1 belong to the border (cyclic) or do not exist.
  double gm1 = 0.0, gm2 = 0.0, dm1 = 0.0, dm2 = 0.0;
  for (int i0 = 0; i0 < M; i0 += kPre) {
    double av[kPre], bv[kPre], cv[kPre], dv[kPre], ev[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int i = i0 + u;
      av[u] = (i >= 2 && i < M) ? A[i] : 0.0;
      bv[u] = (i >= 1 && i < M) ? B[i] : 0.0;
      cv[u] = (i < M) ? C[i] : 1.0;
      dv[u] = (i + 1 < M) ? D[i] : 0.0;
      ev[u] = (i + 2 < M) ? E[i] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int i = i0 + u;
      if (i >= M) break;
      const double ai = av[u], bi = bv[u], di = dv[u], ei = ev[u];
      const double beta = bi - ai * gm2;                       // step 8.1
      const double alpha = cv[u] - ai * dm2 - beta * gm1;      // step 8.2
      if (!(alpha != 0.0) || !isfinite(alpha)) {
        *status = i + 1;
        return;
      }
      // one division per row (the fp64 division is the slow step of this
      // serial sweep); the page's quotients become products with 1/alpha
      const double ra = 1.0 / alpha;
      const double g = (di - beta * dm1) * ra;                 // step 8.3
      const double dd = ei * ra;                               // step 8.4
      r[i] = ra;
      p[i] = ai * ra;                                          // eps_i = a_i (step 14)
      q[i] = beta * ra;
      gam[i] = g;
      del[i] = dd;
      w0[i] = w1[i] = u0[i] = u1[i] = 0.0;
      gm2 = gm1; gm1 = g;
      dm2 = dm1; dm1 = dd;
    }
  }
  if (!cyclic) return;

  // Border pieces of A = [[E, G], [H^T, B]] (eq. (8)).  G is M x 2 (columns
  // N-2, N-1 of rows 0..M-1), H^T is 2 x M (rows N-2, N-1, columns 0..M-1).
  double* g0 = work;            // G column 0
  double* g1 = work + M;        // G column 1
  double* h0 = work + 2 * M;    // H^T row 0
  double* h1 = work + 3 * M;    // H^T row 1
  for (int i = 0; i < 4 * M; ++i) work[i] = 0.0;
  g0[0] += A[0];                 // row 0: a at column N-2
  g1[0] += B[0];                 //        b at column N-1
  g1[1] += A[1];                 // row 1: a at column N-1
  g0[M - 2] += E[M - 2];         // row N-4: e at column N-2
  g0[M - 1] += D[M - 1];         // row N-3: d at column N-2
  g1[M - 1] += E[M - 1];         //          e at column N-1
  h0[N - 4] += A[N - 2];         // row N-2: a at N-4, b at N-3, e at column 0
  h0[N - 3] += B[N - 2];
  h0[0] += E[N - 2];
  h1[N - 3] += A[N - 1];         // row N-1: a at N-3, d at column 0, e at column 1
  h1[0] += D[N - 1];
  h1[1] += E[N - 1];
  const double B00 = C[N - 2], B01 = D[N - 2], B10 = B[N - 1], B11 = C[N - 1];

  // w_k = R^{-T} h_k:  R^T is unit lower with gamma on the first and delta on
  // the second sub-diagonal, so  w_i = h_i - gamma_{i-1} w_{i-1} - delta_{i-2} w_{i-2}.
  // Then h_k^T E^{-1} f = h_k^T R^{-1} L^{-1} f = sum_i w_k,i g_i  with g = L^{-1} f.
  for (int k = 0; k < 2; ++k) {
    const double* h = k ? h1 : h0;
    double* w = k ? w1 : w0;
    double wm1 = 0.0, wm2 = 0.0;
    for (int i0 = 0; i0 < M; i0 += kPre) {
      double hv[kPre], gv[kPre], dv[kPre];
#pragma unroll
      for (int u = 0; u < kPre; ++u) {
        const int i = i0 + u;
        hv[u] = (i < M) ? h[i] : 0.0;
        gv[u] = (i >= 1 && i < M) ? gam[i - 1] : 0.0;
        dv[u] = (i >= 2 && i < M) ? del[i - 2] : 0.0;
      }
#pragma unroll
      for (int u = 0; u < kPre; ++u) {
        const int i = i0 + u;
        if (i >= M) break;
        const double wi = hv[u] - gv[u] * wm1 - dv[u] * wm2;
        w[i] = wi;
        wm2 = wm1; wm1 = wi;
      }
    }
  }
  // u_k = E^{-1} G_k (eq. (11)): forward then back substitution with E's factors.
  for (int k = 0; k < 2; ++k) {
    const double* gcol = k ? g1 : g0;
    double* u = k ? u1 : u0;
    double y1 = 0.0, y2 = 0.0;
    for (int i0 = 0; i0 < M; i0 += kPre) {
      double rv[kPre], fv[kPre], pv[kPre], qv[kPre];
#pragma unroll
      for (int u2 = 0; u2 < kPre; ++u2) {
        const int i = i0 + u2;
        const bool in = i < M;
        rv[u2] = in ? r[i] : 0.0;
        fv[u2] = in ? gcol[i] : 0.0;
        pv[u2] = in ? p[i] : 0.0;
        qv[u2] = in ? q[i] : 0.0;
      }
#pragma unroll
      for (int u2 = 0; u2 < kPre; ++u2) {
        const int i = i0 + u2;
        if (i >= M) break;
        const double y = rv[u2] * fv[u2] - pv[u2] * y2 - qv[u2] * y1;
        u[i] = y;
        y2 = y1; y1 = y;
      }
    }
    double x1 = 0.0, x2 = 0.0;
    for (int i0 = M - 1; i0 >= 0; i0 -= kPre) {
      double yv[kPre], gv[kPre], dv[kPre];
#pragma unroll
      for (int u2 = 0; u2 < kPre; ++u2) {
        const int i = i0 - u2;
        const bool in = i >= 0;
        yv[u2] = in ? u[i] : 0.0;
        gv[u2] = in ? gam[i] : 0.0;
        dv[u2] = in ? del[i] : 0.0;
      }
#pragma unroll
      for (int u2 = 0; u2 < kPre; ++u2) {
        const int i = i0 - u2;
        if (i < 0) break;
        const double x = yv[u2] - gv[u2] * x1 - dv[u2] * x2;
        u[i] = x;
        x2 = x1; x1 = x;
      }
    }
  }
  // S = B - H^T E^{-1} G (eq. (12)) and its inverse.
  double S00 = B00, S01 = B01, S10 = B10, S11 = B11;
#pragma unroll 8
  for (int i = 0; i < M; ++i) {
    S00 -= h0[i] * u0[i];
    S01 -= h0[i] * u1[i];
    S10 -= h1[i] * u0[i];
    S11 -= h1[i] * u1[i];
  }
  const double det = S00 * S11 - S01 * S10;
  if (!(det != 0.0) || !isfinite(det)) {
    *status = M + 1;
    return;
  }
  tail[0] = S11 / det;
  tail[1] = -S01 / det;
  tail[2] = -S10 / det;
  tail[3] = S00 / det;
}

// fp64 table -> fp32 table and double-float (hi, lo) table.
__global__ void k_pack(const double* __restrict__ coef, const double* __restrict__ tail, int n,
                       float* __restrict__ c32, float* __restrict__ t32, float2* __restrict__ cdf,
                       float2* __restrict__ tdf) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  auto split = [](double v) {
    const float hi = __double2float_rn(v);
    const float lo = __double2float_rn(v - (double)hi);
    return make_float2(hi, lo);
  };
  if (i < n) {
    c32[i] = __double2float_rn(coef[i]);
    cdf[i] = split(coef[i]);
  }
  if (i < kTailCount) {
    t32[i] = __double2float_rn(tail[i]);
    tdf[i] = split(tail[i]);
  }
}

}  // namespace

cudaError_t factor_shared(const double* d_bands, int N, int cyclic, double* coef64, double* tail64,
                          double* d_work, int* d_status, cudaStream_t st) {
  k_factor_shared<<<1, 1, 0, st>>>(d_bands, N, cyclic, coef64, tail64, d_work, d_status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t pack_coefficients(const double* coef64, const double* tail64, int n_coef, float* coef32,
                              float* tail32, float2* coefdf, float2* taildf, cudaStream_t st) {
  const int n = n_coef > kTailCount ? n_coef : kTailCount;
  k_pack<<<(n + 255) / 256, 256, 0, st>>>(coef64, tail64, n_coef, coef32, tail32, coefdf, taildf);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pent

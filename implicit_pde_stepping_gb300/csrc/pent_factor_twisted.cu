// Tables of the twisted (two-sided) factorisation used by the double-float kernels.
//
// The LR factorisation of "cuPentBatch – A batched pentadiagonal solver for
// NVIDIA GPUs" (factorisation steps 1–14) eliminates downwards from row 0.
// Rows 0..m-1 of that factorisation depend only on rows 0..m-1 of the matrix,
// so the top half of a system can be eliminated on its own.  The same steps
// applied to the reversed matrix (row i <-> M-1-i, band a <-> e, b <-> d)
// eliminate the bottom half upwards.  What is left is a 4x4 system in
// x_{m-2..m+1}: two rows of the top elimination and two of the bottom one.
// Solving it and back-substituting outwards in both halves gives the same
// solution as the one-sided LR solve (the same linear system, eliminated in
// another order), with half the sweep length per thread.
//
// For a cyclic matrix the same is done for its leading (N-2)x(N-2) block E,
// plus the weights q_k = E^{-T} h_k that give h_k^T E^{-1} f = q_k . f during
// the first sweep (Navon's bordering, eqs. (8)–(12)).  One thread, once per plan.
#include <cmath>

#include "pent_internal.cuh"

namespace pent {
namespace {

// band k (0..4 = a..e) of row j of the M x M leading block, or of its reversal
__device__ double bandv(const double* bands, int N, int M, int k, int j, bool rev) {
  const int col = j + k - 2;
  if (col < 0 || col >= M) return 0.0;
  if (!rev) return bands[(size_t)k * N + j];
  return bands[(size_t)(4 - k) * N + (M - 1 - j)];
}

__device__ float2 split(double v) {
  const float hi = __double2float_rn(v);
  return make_float2(hi, __double2float_rn(v - (double)hi));
}

// LR factor rows 0..R-1 of the (reversed) block: alpha, beta, gamma, delta, eps
__device__ bool lr_rows(const double* bands, int N, int M, int R, bool rev, double* al, double* be,
                        double* ga, double* de, double* ep) {
  double gm1 = 0.0, gm2 = 0.0, dm1 = 0.0, dm2 = 0.0;
  for (int j = 0; j < R; ++j) {
    const double a = bandv(bands, N, M, 0, j, rev), b = bandv(bands, N, M, 1, j, rev);
    const double c = bandv(bands, N, M, 2, j, rev), d = bandv(bands, N, M, 3, j, rev);
    const double e = bandv(bands, N, M, 4, j, rev);
    const double beta = b - a * gm2;
    const double alpha = c - a * dm2 - beta * gm1;
    if (!(alpha != 0.0) || !isfinite(alpha)) return false;
    const double g = (d - beta * dm1) / alpha;
    const double dd = e / alpha;
    al[j] = alpha; be[j] = beta; ga[j] = g; de[j] = dd; ep[j] = a;
    gm2 = gm1; gm1 = g;
    dm2 = dm1; dm1 = dd;
  }
  return true;
}

// 4x4 inverse by Gauss-Jordan with partial pivoting; false if singular.
__device__ bool inv4(double A[4][4], double X[4][4]) {
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) X[i][j] = (i == j) ? 1.0 : 0.0;
  for (int c = 0; c < 4; ++c) {
    int p = c;
    for (int r = c + 1; r < 4; ++r)
      if (fabs(A[r][c]) > fabs(A[p][c])) p = r;
    if (!(fabs(A[p][c]) > 1e-300)) return false;
    for (int j = 0; j < 4; ++j) {
      double t = A[c][j]; A[c][j] = A[p][j]; A[p][j] = t;
      t = X[c][j]; X[c][j] = X[p][j]; X[p][j] = t;
    }
    const double iv = 1.0 / A[c][c];
    for (int j = 0; j < 4; ++j) { A[c][j] *= iv; X[c][j] *= iv; }
    for (int r = 0; r < 4; ++r) {
      if (r == c) continue;
      const double f = A[r][c];
      for (int j = 0; j < 4; ++j) { A[r][j] -= f * A[c][j]; X[r][j] -= f * X[c][j]; }
    }
  }
  return true;
}

// work layout (doubles): 5 arrays of M (top LR), 5 of M (bottom LR), 4 of M (border),
// 2 of M (q), 2 of M (u)
__global__ void k_factor_twisted(const double* __restrict__ bands, int N, int cyclic, int m,
                                 float4* __restrict__ tab, double* __restrict__ twist,
                                 double* __restrict__ w, int* __restrict__ status) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  *status = 0;
  const int M = cyclic ? N - 2 : N;
  const int Mb = M - m;
  double *al = w, *be = w + M, *ga = w + 2 * M, *de = w + 3 * M, *ep = w + 4 * M;
  double *bal = w + 5 * M, *bbe = w + 6 * M, *bga = w + 7 * M, *bde = w + 8 * M, *bep = w + 9 * M;
  double *g0 = w + 10 * M, *g1 = w + 11 * M, *h0 = w + 12 * M, *h1 = w + 13 * M;
  double *q0 = w + 14 * M, *q1 = w + 15 * M, *u0 = w + 16 * M, *u1 = w + 17 * M;
  for (int i = 0; i < 8 * M; ++i) w[10 * M + i] = 0.0;
  if (!lr_rows(bands, N, M, M, false, al, be, ga, de, ep) ||
      !lr_rows(bands, N, M, Mb, true, bal, bbe, bga, bde, bep)) {
    *status = 1;
    return;
  }
  // 4x4 twist system in (x_{m-2}, x_{m-1}, x_m, x_{m+1})
  double T[4][4] = {{1.0, ga[m - 2], de[m - 2], 0.0},
                    {0.0, 1.0, ga[m - 1], de[m - 1]},
                    {bde[Mb - 1], bga[Mb - 1], 1.0, 0.0},
                    {0.0, bde[Mb - 2], bga[Mb - 2], 1.0}};
  double Ti[4][4];
  if (!inv4(T, Ti)) {
    *status = 2;
    return;
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) twist[4 * i + j] = Ti[i][j];
  for (int k = 16; k < kTwistCount; ++k) twist[k] = 0.0;

  if (cyclic) {
    const double* A = bands;
    const double* B = bands + N;
    const double* C = bands + 2 * (size_t)N;
    const double* D = bands + 3 * (size_t)N;
    const double* E = bands + 4 * (size_t)N;
    // border of A = [[E, G], [H^T, B]] (eq. (8)): G columns g0, g1; H^T rows h0, h1
    g0[0] += A[0]; g1[0] += B[0]; g1[1] += A[1];
    g0[M - 2] += E[M - 2]; g0[M - 1] += D[M - 1]; g1[M - 1] += E[M - 1];
    h0[N - 4] += A[N - 2]; h0[N - 3] += B[N - 2]; h0[0] += E[N - 2];
    h1[N - 3] += A[N - 1]; h1[0] += D[N - 1]; h1[1] += E[N - 1];
    // q_k = E^{-T} h_k:  R^T z = h (unit lower: gamma, delta), then L^T q = z
    // (upper: alpha on the diagonal, beta_{i+1} and eps_{i+2} above it)
    for (int k = 0; k < 2; ++k) {
      const double* h = k ? h1 : h0;
      double* q = k ? q1 : q0;
      double z1 = 0.0, z2 = 0.0;
      for (int i = 0; i < M; ++i) {
        const double z = h[i] - (i >= 1 ? ga[i - 1] : 0.0) * z1 - (i >= 2 ? de[i - 2] : 0.0) * z2;
        q[i] = z;
        z2 = z1; z1 = z;
      }
      for (int i = M - 1; i >= 0; --i) {
        const double t1 = (i + 1 < M) ? be[i + 1] * q[i + 1] : 0.0;
        const double t2 = (i + 2 < M) ? ep[i + 2] * q[i + 2] : 0.0;
        q[i] = (q[i] - t1 - t2) / al[i];
      }
    }
    // u_k = E^{-1} G_k (eq. (11))
    for (int k = 0; k < 2; ++k) {
      const double* gc = k ? g1 : g0;
      double* u = k ? u1 : u0;
      double y1 = 0.0, y2 = 0.0;
      for (int i = 0; i < M; ++i) {
        const double y = (gc[i] - ep[i] * y2 - be[i] * y1) / al[i];
        u[i] = y;
        y2 = y1; y1 = y;
      }
      double x1 = 0.0, x2 = 0.0;
      for (int i = M - 1; i >= 0; --i) {
        const double x = u[i] - ga[i] * x1 - de[i] * x2;
        u[i] = x;
        x2 = x1; x1 = x;
      }
    }
    // S = B - H^T E^{-1} G (eq. (12))
    double S00 = C[N - 2], S01 = D[N - 2], S10 = B[N - 1], S11 = C[N - 1];
    for (int i = 0; i < M; ++i) {
      S00 -= h0[i] * u0[i]; S01 -= h0[i] * u1[i];
      S10 -= h1[i] * u0[i]; S11 -= h1[i] * u1[i];
    }
    const double det = S00 * S11 - S01 * S10;
    if (!(det != 0.0) || !isfinite(det)) {
      *status = 3;
      return;
    }
    twist[16] = S11 / det; twist[17] = -S01 / det;
    twist[18] = -S10 / det; twist[19] = S00 / det;
  }

  // pack: top rows j = 0..m-1 (global j), bottom rows j = 0..Mb-1 (global M-1-j)
  int reach = 0;
  for (int dir = 0; dir < 2; ++dir) {
    const int R = dir ? Mb : m;
    const double* A_ = dir ? bal : al;
    const double* B_ = dir ? bbe : be;
    const double* G_ = dir ? bga : ga;
    const double* D_ = dir ? bde : de;
    const double* E_ = dir ? bep : ep;
    for (int j = 0; j < R; ++j) {
      const int gi = dir ? (M - 1 - j) : j;
      const double r = 1.0 / A_[j];
      const float2 sr = split(r), sP = split(-E_[j] * r), sQ = split(-B_[j] * r);
      const float2 sC = split(-G_[j]), sD = split(-D_[j]);
      const float2 sq0 = split(cyclic ? q0[gi] : 0.0), sq1 = split(cyclic ? q1[gi] : 0.0);
      const float2 su0 = split(cyclic ? u0[gi] : 0.0), su1 = split(cyclic ? u1[gi] : 0.0);
      float4* row = tab + (size_t)(dir ? m + j : j) * kTwK;
      row[0] = make_float4(sr.x, sr.y, sP.x, sP.y);
      row[1] = make_float4(sQ.x, sQ.y, sC.x, sC.y);
      row[2] = make_float4(sD.x, sD.y, sq0.x, sq0.y);
      row[3] = make_float4(sq1.x, sq1.y, su0.x, su0.y);
      row[4] = make_float4(su1.x, su1.y, 0.f, 0.f);
      if (cyclic) {
        const double mag = fmax(fmax(fabs(q0[gi]), fabs(q1[gi])), fmax(fabs(u0[gi]), fabs(u1[gi])));
        if (!(mag < ldexp(1.0, -60))) reach = max(reach, j + 1);
      }
    }
  }
  twist[20] = (double)reach;
}

}  // namespace

cudaError_t factor_twisted(const double* d_bands, int N, int cyclic, int m, float4* tab,
                           double* twist, double* d_work, int* d_status, cudaStream_t st) {
  k_factor_twisted<<<1, 1, 0, st>>>(d_bands, N, cyclic, m, tab, twist, d_work, d_status);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pent

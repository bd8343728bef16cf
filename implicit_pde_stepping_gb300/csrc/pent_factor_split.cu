// Tables of the partitioned (split-within-system) double-float kernel.
//
// The LR factors are those of "cuPentBatch – A batched pentadiagonal solver
// for NVIDIA GPUs" (factorisation steps 1–14).  The solve splits each system
// into chunks of L rows handled by different threads (a SPIKE-style
// partitioned solve): every chunk runs the forward and back substitution
// locally with zero boundary values, and the exact solution differs from that
// local one by a combination of four homogeneous solutions per chunk:
//   x = x_local + M1 s0 + M2 s1 + K1 t0 + K2 t1,
// s = (g_{a-2}, g_{a-1}) entering the chunk, t = (x_b, x_{b+1}) leaving it.
// The homogeneous solutions depend only on the matrix, so they are computed
// here once per plan; s and t are found per system by a short scan over the
// chunks.  Cyclic plans add Navon's bordering (eqs. (8)–(12)): x -= u0 x_t0 +
// u1 x_t1 with u_k = E^{-1} G_k, and x_t = S^{-1}(f_t - H^T y).
#include <cmath>

#include "pent_lr.cuh"

namespace pent {
namespace {

constexpr int kFactorThreads = 256;

// One CTA.  The LR recurrences and the bordering sweeps are serial (thread 0,
// or threads 0 and 1); the chunk responses, the row packing and the chunk
// couplings run one thread per chunk or per row.
// work (doubles): al be ga de ep (5 Mpad), g0 g1 h0 h1 (4 Mpad), u0 u1 (2 Mpad),
// H1 H2 M1 M2 K1 K2 (6 Mpad)
__global__ void __launch_bounds__(kFactorThreads)
    k_factor_split(const double* __restrict__ bands, int N, int cyclic, int L, int Mpad,
                   float4* __restrict__ rowtab, double* __restrict__ chunktab,
                   double* __restrict__ extra, double* __restrict__ w, int* __restrict__ status) {
  __shared__ int s_fail;
  __shared__ double s_B[2][2];
  __shared__ double s_red[kFactorThreads][2 * kSpTmax];
  __shared__ double s_q[2];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int M = cyclic ? N - 2 : N;
  const int P = Mpad / L;
  double *al = w, *be = w + Mpad, *ga = w + 2 * Mpad, *de = w + 3 * Mpad, *ep = w + 4 * Mpad;
  double *g0 = w + 5 * Mpad, *g1 = w + 6 * Mpad, *h0 = w + 7 * Mpad, *h1 = w + 8 * Mpad;
  double *u0 = w + 9 * Mpad, *u1 = w + 10 * Mpad;
  double *H1 = w + 11 * Mpad, *H2 = w + 12 * Mpad, *M1 = w + 13 * Mpad, *M2 = w + 14 * Mpad;
  double *K1 = w + 15 * Mpad, *K2 = w + 16 * Mpad;
  if (tid == 0) {
    *status = 0;
    s_fail = lr::factor_rows(bands, N, M, M, false, al, be, ga, de, ep) ? 0 : 1;
  }
  __syncthreads();
  if (s_fail) {
    if (tid == 0) *status = 1;
    return;
  }
  // recurrence coefficients, padding rows decoupled (g = r f, y = g)
  auto R_ = [&](int i) { return i < M ? 1.0 / al[i] : 1.0; };
  auto P_ = [&](int i) { return i < M ? -ep[i] / al[i] : 0.0; };
  auto Q_ = [&](int i) { return i < M ? -be[i] / al[i] : 0.0; };
  auto C_ = [&](int i) { return i < M ? -ga[i] : 0.0; };
  auto D_ = [&](int i) { return i < M ? -de[i] : 0.0; };
  for (int i = tid; i < Mpad; i += nt) u0[i] = u1[i] = 0.0;

  for (int c = tid; c < P; c += nt) {
    const int a = c * L, b = a + L;
    // forward responses to the incoming state (1,0) and (0,1)
    for (int k = 0; k < 2; ++k) {
      double* H = k ? H2 : H1;
      double hm2 = k ? 0.0 : 1.0, hm1 = k ? 1.0 : 0.0;
      for (int j = a; j < b; ++j) {
        const double h = P_(j) * hm2 + Q_(j) * hm1;
        H[j] = h;
        hm2 = hm1; hm1 = h;
      }
    }
    // their local back substitution, and the backward responses to (1,0), (0,1)
    for (int k = 0; k < 2; ++k) {
      const double* H = k ? H2 : H1;
      double* Mv = k ? M2 : M1;
      double* Kv = k ? K2 : K1;
      double m1 = 0.0, m2 = 0.0;
      double k1 = k ? 0.0 : 1.0, k2 = k ? 1.0 : 0.0;   // K at rows b, b+1
      for (int j = b - 1; j >= a; --j) {
        const double mv = H[j] + C_(j) * m1 + D_(j) * m2;
        Mv[j] = mv;
        m2 = m1; m1 = mv;
        const double kv = C_(j) * k1 + D_(j) * k2;
        Kv[j] = kv;
        k2 = k1; k1 = kv;
      }
    }
    double* ct = chunktab + (size_t)c * kSpChunk;
    ct[0] = H1[b - 2]; ct[1] = H2[b - 2]; ct[2] = H1[b - 1]; ct[3] = H2[b - 1];
    ct[4] = M1[a]; ct[5] = M2[a]; ct[6] = M1[a + 1]; ct[7] = M2[a + 1];
    ct[8] = K1[a]; ct[9] = K2[a]; ct[10] = K1[a + 1]; ct[11] = K2[a + 1];
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < kSpExtra; ++k) extra[k] = 0.0;

  if (cyclic) {
    if (tid == 0) {
      double Bm[2][2];
      lr::border(bands, N, g0, g1, h0, h1, Bm);
      s_B[0][0] = Bm[0][0]; s_B[0][1] = Bm[0][1]; s_B[1][0] = Bm[1][0]; s_B[1][1] = Bm[1][1];
    }
    __syncthreads();
    // u_k = E^{-1} G_k (eq. (11)), one thread per column
    if (tid < 2) {
      const int k = tid;
      const double* gc = k ? g1 : g0;
      double* u = k ? u1 : u0;
      // blocks of 8 rows, inputs loaded ahead (one memory wait per block)
      constexpr int kPre = 8;
      double y1 = 0.0, y2 = 0.0;
      for (int i0 = 0; i0 < M; i0 += kPre) {
        double fv[kPre], ev[kPre], bv[kPre], av[kPre];
#pragma unroll
        for (int q2 = 0; q2 < kPre; ++q2) {
          const int i = i0 + q2;
          const bool in = i < M;
          fv[q2] = in ? gc[i] : 0.0;
          ev[q2] = in ? ep[i] : 0.0;
          bv[q2] = in ? be[i] : 0.0;
          av[q2] = in ? 1.0 / al[i] : 1.0;         // off the recurrence's chain
        }
#pragma unroll
        for (int q2 = 0; q2 < kPre; ++q2) {
          const int i = i0 + q2;
          if (i >= M) break;
          const double y = (fv[q2] - ev[q2] * y2 - bv[q2] * y1) * av[q2];
          u[i] = y;
          y2 = y1; y1 = y;
        }
      }
      double x1 = 0.0, x2 = 0.0;
      for (int i0 = M - 1; i0 >= 0; i0 -= kPre) {
        double yv[kPre], gv[kPre], dv[kPre];
#pragma unroll
        for (int q2 = 0; q2 < kPre; ++q2) {
          const int i = i0 - q2;
          const bool in = i >= 0;
          yv[q2] = in ? u[i] : 0.0;
          gv[q2] = in ? ga[i] : 0.0;
          dv[q2] = in ? de[i] : 0.0;
        }
#pragma unroll
        for (int q2 = 0; q2 < kPre; ++q2) {
          const int i = i0 - q2;
          if (i < 0) break;
          const double x = yv[q2] - gv[q2] * x1 - dv[q2] * x2;
          u[i] = x;
          x2 = x1; x1 = x;
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      // S = B - H^T E^{-1} G (eq. (12))
      double S00 = s_B[0][0], S01 = s_B[0][1], S10 = s_B[1][0], S11 = s_B[1][1];
#pragma unroll 8
      for (int i = 0; i < M; ++i) {
        S00 -= h0[i] * u0[i]; S01 -= h0[i] * u1[i];
        S10 -= h1[i] * u0[i]; S11 -= h1[i] * u1[i];
      }
      const double det = S00 * S11 - S01 * S10;
      if (!(det != 0.0) || !isfinite(det)) {
        s_fail = 3;
      } else {
        extra[0] = S11 / det; extra[1] = -S01 / det; extra[2] = -S10 / det; extra[3] = S00 / det;
        // H^T y needs y at rows 0, 1, M-2, M-1 only (N >= 6 keeps them distinct)
        extra[4] = h0[M - 2]; extra[5] = h0[M - 1]; extra[6] = h0[0];
        extra[7] = h1[M - 1]; extra[8] = h1[0]; extra[9] = h1[1];
        extra[10] = M1[M - 2]; extra[11] = M2[M - 2]; extra[12] = M1[M - 1]; extra[13] = M2[M - 1];
        extra[14] = K1[M - 2]; extra[15] = K2[M - 2]; extra[16] = K1[M - 1]; extra[17] = K2[M - 1];
      }
    }
    __syncthreads();
    if (s_fail) {
      if (tid == 0) *status = s_fail;
      return;
    }
  }

  for (int i = tid; i < Mpad; i += nt) {
    const float2 r = lr::split(R_(i)), p = lr::split(P_(i)), q = lr::split(Q_(i));
    const float2 cc = lr::split(C_(i)), d = lr::split(D_(i));
    const float2 m1 = lr::split(M1[i]), m2 = lr::split(M2[i]);
    const float2 k1 = lr::split(K1[i]), k2 = lr::split(K2[i]);
    const float2 a0 = lr::split(u0[i]), a1 = lr::split(u1[i]);
    float4* row = rowtab + (size_t)i * kSpK;
    row[0] = make_float4(r.x, r.y, p.x, p.y);
    row[1] = make_float4(q.x, q.y, a0.x, a0.y);
    row[2] = make_float4(cc.x, cc.y, d.x, d.y);
    row[3] = make_float4(m1.x, m1.y, m2.x, m2.y);
    row[4] = make_float4(k1.x, k1.y, k2.x, k2.y);
    row[5] = make_float4(a1.x, a1.y, 0.f, 0.f);
  }

  // Chunk couplings: products of the boundary maps, and the number T of them
  // that the parallel scan keeps.  Chunks farther apart than T are coupled by
  // products whose summed infinity norm is below 2^-64; those terms are
  // dropped.  If no T <= kSpTmax achieves that, T = 0 selects the exact
  // serial scan.
  auto mul = [](const double* A, const double* B, double* C) {
    const double c0 = A[0] * B[0] + A[1] * B[2], c1 = A[0] * B[1] + A[1] * B[3];
    const double c2 = A[2] * B[0] + A[3] * B[2], c3 = A[2] * B[1] + A[3] * B[3];
    C[0] = c0; C[1] = c1; C[2] = c2; C[3] = c3;
  };
  auto nrm = [](const double* A) { return fmax(fabs(A[0]) + fabs(A[1]), fabs(A[2]) + fabs(A[3])); };
  const double tiny = ldexp(1.0, -64);
  // Products are formed explicitly up to kCap maps; beyond that the remaining
  // terms are bounded geometrically by the largest map norm q (< 1 needed).
  constexpr int kCap = 64;
  double qa = 0.0, qb = 0.0;
  for (int c = tid; c < P; c += nt) {
    qa = fmax(qa, nrm(chunktab + (size_t)c * kSpChunk));
    qb = fmax(qb, nrm(chunktab + (size_t)c * kSpChunk + 8));
  }
  s_red[tid][0] = qa;
  s_red[tid][1] = qb;
  __syncthreads();
  if (tid == 0) {
    for (int k = 1; k < nt; ++k) {
      qa = fmax(qa, s_red[k][0]);
      qb = fmax(qb, s_red[k][1]);
    }
    s_q[0] = qa;
    s_q[1] = qb;
  }
  __syncthreads();
  qa = s_q[0];
  qb = s_q[1];
  const double inf = (double)INFINITY;
  double ta[kSpTmax + 1], tb[kSpTmax + 1];
  for (int t = 0; t <= kSpTmax; ++t) ta[t] = tb[t] = 0.0;
  for (int c = tid; c < P; c += nt) {
    double* ct = chunktab + (size_t)c * kSpChunk;
    for (int k = 12; k < kSpChunk; ++k) ct[k] = 0.0;
    double sa[kSpTmax + 1], sb[kSpTmax + 1];
    for (int t = 0; t <= kSpTmax; ++t) sa[t] = sb[t] = 0.0;
    // forward: A_{c,k} = Phi_{c-1}..Phi_{c-k+1}, k = 2..c (A_{c,1} = I); the
    // scan keeping T couplings drops sum_{k > T} ||A_{c,k}||
    double Acc[4] = {1.0, 0.0, 0.0, 1.0};
    double n = 1.0;
    const int ka = c < kCap ? c : kCap;
    for (int k = 2; k <= ka; ++k) {
      mul(Acc, chunktab + (size_t)(c - k + 1) * kSpChunk, Acc);
      if (k <= kSpTmax)
        for (int q2 = 0; q2 < 4; ++q2) ct[12 + 4 * (k - 2) + q2] = Acc[q2];
      n = nrm(Acc);
      for (int t = 1; t <= kSpTmax; ++t)
        if (k >= t + 1) sa[t] += n;
    }
    if (c > ka) {                                   // terms k = ka+1..c
      const double rest = qa < 1.0 ? n * qa / (1.0 - qa) : inf;
      for (int t = 1; t <= kSpTmax; ++t) sa[t] += rest;
    }
    // backward: B_{c,k} = Kst_{c+1}..Kst_{c+k}, k = 1..P-2-c (B_{c,0} = I);
    // dropped: sum_{k >= T} ||B_{c,k}||
    double Bcc[4] = {1.0, 0.0, 0.0, 1.0};
    n = 1.0;
    const int kbmax = P - 2 - c;
    const int kb = kbmax < kCap ? kbmax : kCap;
    for (int k = 1; k <= kb; ++k) {
      mul(Bcc, chunktab + (size_t)(c + k) * kSpChunk + 8, Bcc);
      if (k <= kSpTmax - 1)
        for (int q2 = 0; q2 < 4; ++q2) ct[24 + 4 * (k - 1) + q2] = Bcc[q2];
      n = nrm(Bcc);
      for (int t = 1; t <= kSpTmax; ++t)
        if (k >= t) sb[t] += n;
    }
    if (kbmax > kb) {
      const double rest = qb < 1.0 ? n * qb / (1.0 - qb) : inf;
      for (int t = 1; t <= kSpTmax; ++t) sb[t] += rest;
    }
    for (int t = 1; t <= kSpTmax; ++t) {
      ta[t] = fmax(ta[t], sa[t]);
      tb[t] = fmax(tb[t], sb[t]);
    }
  }
  __syncthreads();
  for (int t = 1; t <= kSpTmax; ++t) {
    s_red[tid][2 * (t - 1)] = ta[t];
    s_red[tid][2 * (t - 1) + 1] = tb[t];
  }
  __syncthreads();
  if (tid == 0) {
    int T = 0;
    for (int t = 1; t <= kSpTmax && T == 0; ++t) {
      double a = 0.0, b = 0.0;
      for (int k = 0; k < nt; ++k) {
        a = fmax(a, s_red[k][2 * (t - 1)]);
        b = fmax(b, s_red[k][2 * (t - 1) + 1]);
      }
      if (a <= tiny && b <= tiny) T = t;
    }
    extra[18] = (double)T;
    // Border reach: U = E^{-1} G decays away from the two ends of the block;
    // chunks farther than extra[19] chunks from the first (chunk 0) and the last
    // real chunk have every |U| entry below 2^-60 and skip the x_t correction.
    extra[19] = 0.0;
    if (cyclic) {
      const int clast = (M - 1) / L;
      int reach = 0;
      for (int c = 0; c <= clast; ++c) {
        double um = 0.0;
        for (int i = c * L; i < c * L + L && i < M; ++i) um = fmax(um, fmax(fabs(u0[i]), fabs(u1[i])));
        if (!(um < ldexp(1.0, -60))) {
          const int d = min(c, clast - c) + 1;
          reach = max(reach, d);
        }
      }
      extra[19] = (double)reach;
    }
  }
}

}  // namespace

cudaError_t factor_split(const double* d_bands, int N, int cyclic, int L, int Mpad, float4* rowtab,
                         double* chunktab, double* extra, double* d_work, int* d_status,
                         cudaStream_t st) {
  k_factor_split<<<1, kFactorThreads, 0, st>>>(d_bands, N, cyclic, L, Mpad, rowtab, chunktab, extra,
                                               d_work, d_status);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pent

// Per-system matrices: factor + solve in one kernel, one thread per system.
//
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs", the Rewrite
// variant (a new matrix at every call): factorisation steps 1–14 fused with the
// forward substitution in one sweep down the rows, then back substitution up
// the rows.  Diagonally dominant or SPD matrices need no pivoting (the page's
// stability remark), so none is done; a zero or non-finite pivot is reported
// per system in `info`.
//
// The page overwrites the bands with the factors.  Here the bands are inputs
// and stay unchanged: gamma_i and delta_i go to the caller's scratch `work`
// (two interleaved [N][batch] arrays), and g is written over the right-hand
// side in place, read back by the backward sweep.
//
// Layouts of the bands and the right-hand side: interleaved [N][batch], or
// block-interleaved with blocks of bs systems ((i, s) at (s / bs) N bs +
// i bs + s % bs); the scratch stays interleaved.
#include "df64.cuh"
#include "pent_internal.cuh"

namespace pent {
namespace {

using df::D2;

constexpr int kThreads = 128;
constexpr int kUnroll = 4;

template <typename T>
__global__ void __launch_bounds__(kThreads)
    k_persys_thread(const T* __restrict__ A, const T* __restrict__ B, const T* __restrict__ C,
                    const T* __restrict__ D, const T* __restrict__ E, T* __restrict__ X,
                    T* __restrict__ Wg, T* __restrict__ Wd, int N, int batch, int bs, int* __restrict__ info) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const size_t ld = bs ? (size_t)bs : (size_t)batch;                          // row stride of the data
  const size_t sb = bs ? (size_t)(s / bs) * N * bs + s % bs : (size_t)s;     // row 0 of system s
  const size_t lw = (size_t)batch;                                             // scratch: interleaved
  T gm1 = T(0), gm2 = T(0), dm1 = T(0), dm2 = T(0), g1 = T(0), g2 = T(0);
  int bad = 0;
  for (int i0 = 0; i0 < N; i0 += kUnroll) {
    T a[kUnroll], b[kUnroll], c[kUnroll], d[kUnroll], e[kUnroll], f[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      const size_t o = (size_t)i * ld + sb;
      const bool in = i < N;
      a[u] = (in && i >= 2) ? A[o] : T(0);
      b[u] = (in && i >= 1) ? B[o] : T(0);
      c[u] = in ? C[o] : T(1);
      d[u] = (in && i + 1 < N) ? D[o] : T(0);
      e[u] = (in && i + 2 < N) ? E[o] : T(0);
      f[u] = in ? X[o] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < N) {
        const size_t o = (size_t)i * ld + sb, ow = (size_t)i * lw + s;
        const T beta = b[u] - a[u] * gm2;
        const T alpha = c[u] - a[u] * dm2 - beta * gm1;
        if (bad == 0 && !(alpha != T(0) && isfinite(alpha))) bad = i + 1;
        const T ra = T(1) / alpha;
        const T gam = (d[u] - beta * dm1) * ra;
        const T del = e[u] * ra;
        const T g = (f[u] - a[u] * g2 - beta * g1) * ra;
        Wg[ow] = gam;
        Wd[ow] = del;
        X[o] = g;
        gm2 = gm1; gm1 = gam;
        dm2 = dm1; dm1 = del;
        g2 = g1; g1 = g;
      }
    }
  }
  T x1 = T(0), x2 = T(0);
  for (int i0 = N - 1; i0 >= 0; i0 -= kUnroll) {
    T gv[kUnroll], gm[kUnroll], dl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      const size_t o = (size_t)(i >= 0 ? i : 0) * ld + sb, ow = (size_t)(i >= 0 ? i : 0) * lw + s;
      gv[u] = (i >= 0) ? X[o] : T(0);
      gm[u] = (i >= 0) ? Wg[ow] : T(0);
      dl[u] = (i >= 0) ? Wd[ow] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      if (i >= 0) {
        const T x = gv[u] - gm[u] * x1 - dl[u] * x2;
        X[(size_t)i * ld + sb] = x;
        x2 = x1;
        x1 = x;
      }
    }
  }
  if (info) info[s] = bad;
}

// ---------------------------------------------------------------------------
// fp64 matrices in double-float: the same sweeps with every value an
// unevaluated pair of floats on the FP32 pipe (the fp64 pipe runs at ~1/70 of
// it), fp64 inputs and outputs converted by integer operations; gamma, delta
// and g go to the scratch and the right-hand side as (hi, lo) pairs, the same
// 8 bytes as a double.
// ---------------------------------------------------------------------------

// 1/a: the float reciprocal refined by one Newton–Raphson step,
// r = r0 + r0 (1 - a r0), with a r0 formed exactly (relative error ~2^-46)
__device__ __forceinline__ D2 df_recip(D2 a) {
  const float r0 = __frcp_rn(a.h);
  float p, pe;
  df::two_prod(a.h, r0, p, pe);
  const float e = __fmaf_rn(-a.l, r0, __fsub_rn(__fsub_rn(1.f, p), pe));
  return D2{r0, r0 * e};
}
__device__ __forceinline__ D2 dneg(D2 a) { return D2{-a.h, -a.l}; }
__device__ __forceinline__ float2 f2(D2 a) { return make_float2(a.h, a.l); }
__device__ __forceinline__ D2 d2(float2 a) { return D2{a.x, a.y}; }

__global__ void __launch_bounds__(kThreads)
    k_persys_thread_df(const double* __restrict__ A, const double* __restrict__ B, const double* __restrict__ C,
                       const double* __restrict__ D, const double* __restrict__ E, double* __restrict__ X,
                       float2* __restrict__ Wg, float2* __restrict__ Wd, int N, int batch, int bs,
                       int* __restrict__ info) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const size_t ld = bs ? (size_t)bs : (size_t)batch;                          // row stride of the data
  const size_t sb = bs ? (size_t)(s / bs) * N * bs + s % bs : (size_t)s;     // row 0 of system s
  const size_t lw = (size_t)batch;                                             // scratch: interleaved
  float2* Xg = reinterpret_cast<float2*>(X);                                   // g as (hi, lo) in place
  const D2 z{0.f, 0.f};
  D2 gm1 = z, gm2 = z, dm1 = z, dm2 = z, g1 = z, g2 = z;
  int bad = 0;
  for (int i0 = 0; i0 < N; i0 += kUnroll) {
    double a[kUnroll], b[kUnroll], c[kUnroll], d[kUnroll], e[kUnroll], f[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      const size_t o = (size_t)i * ld + sb;
      const bool in = i < N;
      a[u] = (in && i >= 2) ? A[o] : 0.0;
      b[u] = (in && i >= 1) ? B[o] : 0.0;
      c[u] = in ? C[o] : 1.0;
      d[u] = (in && i + 1 < N) ? D[o] : 0.0;
      e[u] = (in && i + 2 < N) ? E[o] : 0.0;
      f[u] = in ? X[o] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < N) {
        const size_t o = (size_t)i * ld + sb, ow = (size_t)i * lw + s;
        const D2 ai = df::from_double(a[u]), bi = df::from_double(b[u]), ci = df::from_double(c[u]);
        const D2 na = dneg(ai);
        const D2 beta = df::axpy(bi, na, gm2);
        const D2 alpha = df::sum3(ci, na, dm2, dneg(beta), gm1);
        if (bad == 0 && !(alpha.h != 0.f && isfinite(alpha.h))) bad = i + 1;
        const D2 ra = df_recip(alpha);
        const D2 gam = df::mul(df::axpy(df::from_double(d[u]), dneg(beta), dm1), ra);
        const D2 del = df::mul(df::from_double(e[u]), ra);
        const D2 g = df::mul(df::sum3(df::from_double(f[u]), na, g2, dneg(beta), g1), ra);
        Wg[ow] = f2(gam);
        Wd[ow] = f2(del);
        Xg[o] = f2(g);
        gm2 = gm1; gm1 = gam;
        dm2 = dm1; dm1 = del;
        g2 = g1; g1 = g;
      }
    }
  }
  D2 x1 = z, x2 = z;
  for (int i0 = N - 1; i0 >= 0; i0 -= kUnroll) {
    float2 gv[kUnroll], gm[kUnroll], dl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      const size_t o = (size_t)(i >= 0 ? i : 0) * ld + sb, ow = (size_t)(i >= 0 ? i : 0) * lw + s;
      gv[u] = (i >= 0) ? Xg[o] : make_float2(0.f, 0.f);
      gm[u] = (i >= 0) ? Wg[ow] : make_float2(0.f, 0.f);
      dl[u] = (i >= 0) ? Wd[ow] : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      if (i >= 0) {
        const D2 x = df::sum3(d2(gv[u]), dneg(d2(gm[u])), x1, dneg(d2(dl[u])), x2);
        X[(size_t)i * ld + sb] = df::to_double(x);
        x2 = x1;
        x1 = x;
      }
    }
  }
  if (info) info[s] = bad;
}

template <typename T>
cudaError_t launch(const void* a, const void* b, const void* c, const void* d, const void* e,
                   void* X, int N, int batch, int bs, void* work, int* info, cudaStream_t st) {
  T* Wg = static_cast<T*>(work);
  T* Wd = Wg + (size_t)N * batch;
  const int grid = (batch + kThreads - 1) / kThreads;
  k_persys_thread<T><<<grid, kThreads, 0, st>>>(
      static_cast<const T*>(a), static_cast<const T*>(b), static_cast<const T*>(c),
      static_cast<const T*>(d), static_cast<const T*>(e), static_cast<T*>(X), Wg, Wd, N, batch, bs,
      info);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

size_t persys_work_bytes(int N, int batch, pent_dtype dt) {
  const size_t elem = dt == PENT_F64 ? sizeof(double) : sizeof(float);
  return 2 * (size_t)N * (size_t)batch * elem;
}

cudaError_t persys_thread_df(const void* a, const void* b, const void* c, const void* d, const void* e,
                             void* X, int N, int batch, int bs, void* work, int* info, cudaStream_t st) {
  float2* Wg = static_cast<float2*>(work);
  float2* Wd = Wg + (size_t)N * batch;
  const int grid = (batch + kThreads - 1) / kThreads;
  k_persys_thread_df<<<grid, kThreads, 0, st>>>(
      static_cast<const double*>(a), static_cast<const double*>(b), static_cast<const double*>(c),
      static_cast<const double*>(d), static_cast<const double*>(e), static_cast<double*>(X), Wg, Wd, N,
      batch, bs, info);
  note_launch();
  return cudaGetLastError();
}

cudaError_t persys_thread(const void* a, const void* b, const void* c, const void* d, const void* e,
                          void* X, int N, int batch, int bs, pent_dtype dt, void* work, int* info,
                          cudaStream_t st) {
  if (dt == PENT_F64) return launch<double>(a, b, c, d, e, X, N, batch, bs, work, info, st);
  return launch<float>(a, b, c, d, e, X, N, batch, bs, work, info, st);
}

}  // namespace pent

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
#include "fg.cuh"
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
__device__ __forceinline__ double pair_to_double(float2 a) { return (double)a.x + (double)a.y; }

// v * 2^-(e - 1023) as a pair, off = (e - 127) << 20
__device__ __forceinline__ D2 sdf(double v, uint32_t off) {
  float h, l;
  fg::split(v, off, h, l);
  return D2{h, l};
}

// Native fp64 from row isw on (the double-float sweep stopped there), then the
// back substitution of the whole system in fp64.  Rows before isw hold gamma,
// delta as (hi, lo) pairs and g as a pair times 2^-S (os: the output constant of
// that scale); from isw on the scratch and X hold fp64 values.
__device__ __noinline__ void native_persys_rest(const double* __restrict__ A, const double* __restrict__ B,
                                                const double* __restrict__ C, const double* __restrict__ D,
                                                const double* __restrict__ E, double* __restrict__ X,
                                                float2* __restrict__ Wg, float2* __restrict__ Wd, int N,
                                                size_t ld, size_t sb, size_t lw, int s, int isw, uint32_t os,
                                                bool sset, D2 gm1p, D2 gm2p, D2 dm1p, D2 dm2p, D2 g1p, D2 g2p,
                                                int& bad) {
  double* Wgd = reinterpret_cast<double*>(Wg);
  double* Wdd = reinterpret_cast<double*>(Wd);
  const float2* Xg = reinterpret_cast<const float2*>(X);
  double gm1 = (double)gm1p.h + gm1p.l, gm2 = (double)gm2p.h + gm2p.l;
  double dm1 = (double)dm1p.h + dm1p.l, dm2 = (double)dm2p.h + dm2p.l;
  // before the first nonzero f every g is exactly zero
  double g1 = sset ? fg::join(g1p.h, g1p.l, os) : 0.0, g2 = sset ? fg::join(g2p.h, g2p.l, os) : 0.0;
  if (isw == 0) g1 = g2 = 0.0;
  if (isw == 1) g2 = 0.0;
  for (int i = isw; i < N; ++i) {
    const size_t o = (size_t)i * ld + sb, ow = (size_t)i * lw + s;
    const double a = i >= 2 ? A[o] : 0.0, b = i >= 1 ? B[o] : 0.0, c = C[o];
    const double d = i + 1 < N ? D[o] : 0.0, e = i + 2 < N ? E[o] : 0.0, f = X[o];
    const double beta = b - a * gm2;
    const double alpha = c - a * dm2 - beta * gm1;
    if (bad == 0 && !(alpha != 0.0 && isfinite(alpha))) bad = i + 1;
    const double ra = 1.0 / alpha;
    const double gam = (d - beta * dm1) * ra;
    const double del = e * ra;
    const double g = (f - a * g2 - beta * g1) * ra;
    Wgd[ow] = gam;
    Wdd[ow] = del;
    X[o] = g;
    gm2 = gm1; gm1 = gam;
    dm2 = dm1; dm1 = del;
    g2 = g1; g1 = g;
  }
  double x1 = 0.0, x2 = 0.0;
  for (int i = N - 1; i >= 0; --i) {
    const size_t o = (size_t)i * ld + sb, ow = (size_t)i * lw + s;
    const bool nat = i >= isw;
    const double g = nat ? X[o] : (sset ? fg::join(Xg[o].x, Xg[o].y, os) : 0.0);
    const double gam = nat ? Wgd[ow] : pair_to_double(Wg[ow]);
    const double del = nat ? Wdd[ow] : pair_to_double(Wd[ow]);
    const double x = g - gam * x1 - del * x2;
    X[o] = x;
    x2 = x1;
    x1 = x;
  }
}

// Range.  Row i is scaled by 2^-(e_i - 1023), e_i the exponent field of its
// diagonal entry c_i: scaling a row of A together with f_i leaves gamma, delta,
// g and x unchanged and keeps the row's bands near 1.  The solution scale 2^S
// of the system (g and x are held as pairs times 2^-S) is fixed at its first
// nonzero f_i, from |f_i / c_i|; rows much smaller than that are negligible
// against it.  A row the pairs cannot represent in that scale (|f_i / c_i| more
// than 2^60 above it), a zero, subnormal or non-finite diagonal entry or f_i,
// or a scale outside [2^-890, 2^890], sends the thread to native fp64 from that
// row on: the rows already done are exact in the pair format (f_i is read
// before g_i replaces it), so the sweep continues from them, and the back
// substitution then runs natively over the whole system.  A system whose f is
// zero gets exact zeros.
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
  int S = 0;            // solution-scale exponent (set at the first nonzero f_i)
  bool sset = false;
  int isw = N;          // first row handled natively (N: none)
  for (int i0 = 0; i0 < N && isw == N; i0 += kUnroll) {
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
      if (i < N && isw == N) {
        const uint32_t mc = fg::mag_bits(c[u]), mf = fg::mag_bits(f[u]);
        const uint32_t ec = mc >> 20, ef = mf >> 20;
        bool nat = ec == 0u || ec >= 2047u || ef >= 2047u || (ef == 0u && mf != 0u);
        if (!nat && mf != 0u) {
          const int rel = (int)ef - (int)ec;
          if (!sset) {
            S = rel;
            sset = true;
            nat = rel < -890 || rel > 890;
          } else {
            nat = rel - S > 60;
          }
        }
        if (nat) {
          isw = i;
        } else {
          const size_t o = (size_t)i * ld + sb, ow = (size_t)i * lw + s;
          const uint32_t ob = (ec - 127u) << 20;                 // bands of row i: x 2^-(ec - 1023)
          const uint32_t of = ob + ((uint32_t)S << 20);           // f_i: also x 2^-S
          const D2 ai = sdf(a[u], ob), bi = sdf(b[u], ob), ci = sdf(c[u], ob);
          const D2 na = dneg(ai);
          const D2 beta = df::axpy(bi, na, gm2);
          const D2 alpha = df::sum3(ci, na, dm2, dneg(beta), gm1);
          if (bad == 0 && !(alpha.h != 0.f && isfinite(alpha.h))) bad = i + 1;
          const D2 ra = df_recip(alpha);
          const D2 gam = df::mul(df::axpy(sdf(d[u], ob), dneg(beta), dm1), ra);
          const D2 del = df::mul(sdf(e[u], ob), ra);
          const D2 g = df::mul(df::sum3(sdf(f[u], of), na, g2, dneg(beta), g1), ra);
          Wg[ow] = f2(gam);
          Wd[ow] = f2(del);
          Xg[o] = f2(g);
          gm2 = gm1; gm1 = gam;
          dm2 = dm1; dm1 = del;
          g2 = g1; g1 = g;
        }
      }
    }
  }
  const uint32_t os = ((uint32_t)S + 1023u - 127u) << 20;         // pairs x 2^S back to fp64
  if (isw == N) {
    if (!sset) {                                                  // f = 0: x = 0
      for (int i = 0; i < N; ++i) X[(size_t)i * ld + sb] = 0.0;
    } else {
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
            X[(size_t)i * ld + sb] = fg::join(x.h, x.l, os);
            x2 = x1;
            x1 = x;
          }
        }
      }
    }
  } else {
    native_persys_rest(A, B, C, D, E, X, Wg, Wd, N, ld, sb, lw, s, isw, os, sset, gm1, gm2, dm1, dm2, g1, g2, bad);
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

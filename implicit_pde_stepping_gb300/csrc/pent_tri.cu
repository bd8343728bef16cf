// Batched tridiagonal solves with per-system matrices.
//
// "Simulating the behavior of the human brain on GPUs" (Valero-Lara et al.),
// section 4.1 "Tridiagonal linear systems" and 4.1.1 (cuThomasBatch): the
// Thomas algorithm, one system per thread, systems interleaved in memory so
// that a warp's loads of one row are contiguous.  Rows: a_i below the
// diagonal (column i-1), b_i on it, c_i above it (column i+1).
//
// Layouts: interleaved [N][batch] (element (i, s) at i * batch + s), or the
// page's block-interleaved layout (section 4.1.1) with blocks of bs systems,
// each block an interleaved [N][bs] array: (i, s) at (s / bs) N bs + i bs + s % bs.
// Either way a system's rows are a fixed stride apart from its own base.
//
// Two kernels:
//   k_tri_thread<T>  the page's mapping: forward elimination writes c'_i to a
//                    scratch array and y'_i over the right-hand side, the
//                    backward substitution reads both back.  Any N, fp32/fp64.
//   k_tri_split      fp32, N <= 512: each system is cut into P = 2^k chunks of
//                    L = 16 rows, one thread per chunk, and never leaves
//                    registers, so memory sees the minimum (a, b, c, y read
//                    once, u written once).  Per chunk [s, e] the downward
//                    elimination gives x_i + c'_i x_{i+1} + l_i x_{s-1} = y'_i;
//                    the upward elimination from row e-1, with the chunk's own
//                    last row t_c = x_e as the right unknown, gives
//                        x_i = y''_i - l'_i t_{c-1} - r_i t_c      (i < e).
//                    Row e then reads x_e + l_e t_{c-1} + c'_e x_{s'} = y'_e with
//                    x_{s'} (the next chunk's first row) in the same form, which
//                    leaves one equation per chunk in the t's:
//                        l_e t_{c-1} + (1 - c'_e l'_s') t_c - c'_e r_s' t_{c+1}
//                            = y'_e - c'_e y''_s',
//                    a P-unknown tridiagonal system solved by parallel cyclic
//                    reduction across P lanes with warp shuffles.  Then every row
//                    follows from t_{c-1} and t_c.
//   The partition trades the page's 8n operations for about twice as many,
//   which fp32 affords: the kernel is bound by memory, not arithmetic.
//   A CTA's tile of a, b, c and y (16 systems x all rows) reaches shared memory
//   by TMA: one thread issues four box copies per 256 rows and the CTA waits
//   on an mbarrier, so the whole tile is in flight without holding registers.
//   Where a tensor map cannot describe the arrays (base or row pitch not a
//   multiple of 16 bytes) every thread stages its own rows with 4-byte
//   cp.async instead.
#include "cp_async.cuh"
#include "df64.cuh"
#include "fg.cuh"
#include "pent_internal.cuh"
#include "tma.cuh"

namespace pent {
namespace {

using df::D2;

constexpr int kThreads = 128;
constexpr int kUnroll = 4;

template <typename T>
__device__ __forceinline__ bool bad_pivot(T d) {
  return !(d != T(0)) || !isfinite(d);
}

// 1/x: the fast hardware reciprocal in fp32 (about 1 ulp, well inside the fp32
// tolerance of the solve); IEEE division in fp64
__device__ __forceinline__ float recip(float x) { return __fdividef(1.f, x); }
__device__ __forceinline__ double recip(double x) { return 1.0 / x; }

// ---------------------------------------------------------------------------
// one thread per system (cuThomasBatch mapping)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
    k_tri_thread(const T* __restrict__ A, const T* __restrict__ B, const T* __restrict__ C,
                 T* __restrict__ X, T* __restrict__ Wc, int N, int batch, int bs, int* __restrict__ info) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const size_t ld = bs ? (size_t)bs : (size_t)batch;                          // row stride
  const size_t sb = bs ? (size_t)(s / bs) * N * bs + s % bs : (size_t)s;     // row 0 of system s
  T cp = T(0), yp = T(0);
  int bad = 0;
  for (int i0 = 0; i0 < N; i0 += kUnroll) {
    T a[kUnroll], b[kUnroll], c[kUnroll], y[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      const size_t o = (size_t)i * ld + sb;
      const bool in = i < N;
      a[u] = (in && i >= 1) ? A[o] : T(0);
      b[u] = in ? B[o] : T(1);
      c[u] = (in && i + 1 < N) ? C[o] : T(0);
      y[u] = in ? X[o] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < N) {
        const size_t o = (size_t)i * ld + sb;
        const T den = b[u] - cp * a[u];
        if (bad == 0 && bad_pivot(den)) bad = i + 1;
        const T rd = recip(den);
        cp = c[u] * rd;
        yp = (y[u] - yp * a[u]) * rd;
        Wc[o] = cp;
        X[o] = yp;
      }
    }
  }
  T x1 = T(0);
  for (int i0 = N - 1; i0 >= 0; i0 -= kUnroll) {
    T yv[kUnroll], cv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      const size_t o = (size_t)(i >= 0 ? i : 0) * ld + sb;
      yv[u] = (i >= 0) ? X[o] : T(0);
      cv[u] = (i >= 0) ? Wc[o] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 - u;
      if (i >= 0) {
        const T x = yv[u] - cv[u] * x1;
        X[(size_t)i * ld + sb] = x;
        x1 = x;
      }
    }
  }
  if (info) info[s] = bad;
}

// ---------------------------------------------------------------------------
// fp64 systems in double-float, one thread per system: the same Thomas sweeps
// with every value an unevaluated pair of floats on the FP32 pipe (the fp64
// pipe runs at ~1/70 of it), fp64 inputs and outputs converted by integer
// operations; c' goes to the scratch and y' over the right-hand side as
// (hi, lo) pairs, the same 8 bytes as a double.
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

// Range, as in the per-system pentadiagonal kernel: row i scaled by the power
// of two of its diagonal b_i (c' and y' are unchanged), the solution scale 2^S
// fixed at the first nonzero y_i from |y_i / b_i|, and native fp64 from the
// first row the pairs cannot represent in that scale (more than 2^60 above it;
// zero, subnormal or non-finite b_i or y_i; S outside [2^-890, 2^890]).  A zero
// right-hand side gives exact zeros.
__device__ __forceinline__ D2 tsdf(double v, uint32_t off) {
  float h, l;
  fg::split(v, off, h, l);
  return D2{h, l};
}

__device__ __noinline__ void native_tri_rest(const double* __restrict__ A, const double* __restrict__ B,
                                             const double* __restrict__ C, double* __restrict__ X,
                                             float2* __restrict__ Wc, int N, int batch, size_t ld, size_t sb,
                                             int s, int isw, uint32_t os, bool sset, D2 cpp, D2 ypp, int& bad) {
  double* Wcd = reinterpret_cast<double*>(Wc);
  const float2* Xp = reinterpret_cast<const float2*>(X);
  double cp = (double)cpp.h + cpp.l;
  double yp = (sset && isw > 0) ? fg::join(ypp.h, ypp.l, os) : 0.0;
  if (isw == 0) cp = 0.0;
  for (int i = isw; i < N; ++i) {
    const size_t o = (size_t)i * ld + sb, ow = (size_t)i * batch + s;
    const double a = i >= 1 ? A[o] : 0.0, b = B[o], c = i + 1 < N ? C[o] : 0.0, y = X[o];
    const double den = b - cp * a;
    if (bad == 0 && !(den != 0.0 && isfinite(den))) bad = i + 1;
    const double rd = 1.0 / den;
    cp = c * rd;
    yp = (y - yp * a) * rd;
    Wcd[ow] = cp;
    X[o] = yp;
  }
  double x1 = 0.0;
  for (int i = N - 1; i >= 0; --i) {
    const size_t o = (size_t)i * ld + sb, ow = (size_t)i * batch + s;
    const bool nat = i >= isw;
    const double y = nat ? X[o] : (sset ? fg::join(Xp[o].x, Xp[o].y, os) : 0.0);
    const double c = nat ? Wcd[ow] : (double)Wc[ow].x + (double)Wc[ow].y;
    const double x = y - c * x1;
    X[o] = x;
    x1 = x;
  }
}

__global__ void __launch_bounds__(kThreads)
    k_tri_thread_df(const double* __restrict__ A, const double* __restrict__ B, const double* __restrict__ C,
                    double* __restrict__ X, float2* __restrict__ Wc, int N, int batch, int bs,
                    int* __restrict__ info) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const size_t ld = bs ? (size_t)bs : (size_t)batch;                          // row stride
  const size_t sb = bs ? (size_t)(s / bs) * N * bs + s % bs : (size_t)s;     // row 0 of system s
  float2* Xp = reinterpret_cast<float2*>(X);                                   // y' as (hi, lo) in place
  D2 cp{0.f, 0.f}, yp{0.f, 0.f};
  int bad = 0;
  int S = 0;            // solution-scale exponent (set at the first nonzero y_i)
  bool sset = false;
  int isw = N;          // first row handled natively (N: none)
  for (int i0 = 0; i0 < N && isw == N; i0 += kUnroll) {
    double a[kUnroll], b[kUnroll], c[kUnroll], y[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      const size_t o = (size_t)i * ld + sb;
      const bool in = i < N;
      a[u] = (in && i >= 1) ? A[o] : 0.0;
      b[u] = in ? B[o] : 1.0;
      c[u] = (in && i + 1 < N) ? C[o] : 0.0;
      y[u] = in ? X[o] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u;
      if (i < N && isw == N) {
        const uint32_t mb = fg::mag_bits(b[u]), my = fg::mag_bits(y[u]);
        const uint32_t eb = mb >> 20, ey = my >> 20;
        bool nat = eb == 0u || eb >= 2047u || ey >= 2047u || (ey == 0u && my != 0u);
        if (!nat && my != 0u) {
          const int rel = (int)ey - (int)eb;
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
          const size_t o = (size_t)i * ld + sb;
          const uint32_t ob = (eb - 127u) << 20;                 // row i: x 2^-(eb - 1023)
          const uint32_t oy = ob + ((uint32_t)S << 20);           // y_i: also x 2^-S
          const D2 na = df::neg(tsdf(a[u], ob));
          const D2 den = df::axpy(tsdf(b[u], ob), na, cp);
          if (bad == 0 && !(den.h != 0.f && isfinite(den.h))) bad = i + 1;
          const D2 rd = df_recip(den);
          cp = df::mul(tsdf(c[u], ob), rd);
          yp = df::mul(df::axpy(tsdf(y[u], oy), na, yp), rd);
          Wc[(size_t)i * batch + s] = make_float2(cp.h, cp.l);
          Xp[o] = make_float2(yp.h, yp.l);
        }
      }
    }
  }
  const uint32_t os = ((uint32_t)S + 1023u - 127u) << 20;         // pairs x 2^S back to fp64
  if (isw == N) {
    if (!sset) {                                                  // y = 0: x = 0
      for (int i = 0; i < N; ++i) X[(size_t)i * ld + sb] = 0.0;
    } else {
      D2 x1{0.f, 0.f};
      for (int i0 = N - 1; i0 >= 0; i0 -= kUnroll) {
        float2 yv[kUnroll], cv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = i0 - u;
          const int ii = i >= 0 ? i : 0;
          yv[u] = (i >= 0) ? Xp[(size_t)ii * ld + sb] : make_float2(0.f, 0.f);
          cv[u] = (i >= 0) ? Wc[(size_t)ii * batch + s] : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = i0 - u;
          if (i >= 0) {
            const D2 x = df::axpy(D2{yv[u].x, yv[u].y}, df::neg(D2{cv[u].x, cv[u].y}), x1);
            X[(size_t)i * ld + sb] = fg::join(x.h, x.l, os);
            x1 = x;
          }
        }
      }
    }
  } else {
    native_tri_rest(A, B, C, X, Wc, N, batch, ld, sb, s, isw, os, sset, cp, yp, bad);
  }
  if (info) info[s] = bad;
}

// ---------------------------------------------------------------------------
// partitioned fp32 kernel: 16 systems x P chunks of L rows per CTA (3 CTAs/SM up to
// N = 256, so that one CTA's tile load overlaps the others' arithmetic and barriers)
// ---------------------------------------------------------------------------
constexpr int kTriSB = 16;    // systems per CTA

struct TriMaps {
  CUtensorMap m[4];   // a, b, c, y
};

// Staged tile: TMA layout [array][RS rows][SB systems]; cp.async layout
// [array][L rows][SB * P threads].
template <int L, int P, bool TMA>
__global__ void __launch_bounds__(kTriSB * P, P <= 16 ? 3 : 1)
    k_tri_split(const __grid_constant__ TriMaps maps, const float* __restrict__ A,
                const float* __restrict__ B, const float* __restrict__ C, float* __restrict__ X, int N,
                int batch, int bs, int RS, int BR, int* __restrict__ info) {
  constexpr int SB = kTriSB;
  // Per chunk: first row (l', r, y''), last row (l', r, y''); t_c = x at the last row.
  // Stored [quantity][chunk][system] with rows of SB + 1 so that both thread
  // mappings (threads over systems; threads over chunks) spread over the banks.
  __shared__ float sB[6][P][SB + 1];
  __shared__ float sT[P][SB + 1];
  __shared__ int sBad[SB];
  constexpr int NT = SB * P;
  extern __shared__ __align__(128) float stage[];
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  const int lane = threadIdx.x % SB;         // phases 1, 3: system of this thread
  const int c = threadIdx.x / SB;            //              its chunk
  const int s = blockIdx.x * SB + lane;
  const bool act = s < batch;
  const size_t ld = bs ? (size_t)bs : (size_t)batch;                          // row stride
  const size_t sb = bs ? (size_t)(s / bs) * N * bs + s % bs : (size_t)s;     // row 0 of system s
  const int row0 = c * L;
  if (threadIdx.x < SB) sBad[threadIdx.x] = 0;

  int bad = 0;
  // ---- 0. the tile into shared memory, all of it in flight at once
  if constexpr (TMA) {
    if (tid == 0) tma::mbar_init(&bar, 1);
    __syncthreads();
    if (tid == 0) {
      tma::mbar_expect_tx(&bar, (unsigned)(4 * RS * SB * sizeof(float)));
      for (int arr = 0; arr < 4; ++arr)
        for (int y0 = 0; y0 < RS; y0 += BR) {
          float* dst = stage + ((size_t)arr * RS + y0) * SB;
          if (bs) tma::load_3d(dst, &maps.m[arr], (blockIdx.x * SB) % bs, y0, (blockIdx.x * SB) / bs, &bar);
          else tma::load_2d(dst, &maps.m[arr], blockIdx.x * SB, y0, &bar);
        }
    }
    if (!tma::mbar_wait(&bar, 0, 2000000000ull)) bad = -1;   // 2 s: the copy never arrived
  } else {
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const int i = row0 + j;
      if (act && i < N) {
        const size_t o = (size_t)i * ld + sb;
        cp_async4(&stage[(0 * L + j) * NT + tid], A + o);
        cp_async4(&stage[(1 * L + j) * NT + tid], B + o);
        cp_async4(&stage[(2 * L + j) * NT + tid], C + o);
        cp_async4(&stage[(3 * L + j) * NT + tid], X + o);
      }
    }
    cp_async_wait_all();
  }
  auto staged = [&](int arr, int j) -> float {
    return TMA ? stage[((size_t)arr * RS + row0 + j) * SB + lane] : stage[(arr * L + j) * NT + tid];
  };

  // ---- 1. downward elimination: x_i + c'_i x_{i+1} + l_i x_{s-1} = y'_i
  float cp[L], lv[L], yv[L];
  {
    float cprev = 0.f, lprev = 0.f, yprev = 0.f;
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const int i = row0 + j;
      const bool in = act && i < N;
      const float a = (in && i >= 1) ? staged(0, j) : 0.f;
      const float b = in ? staged(1, j) : 1.f;
      const float cc = (in && i + 1 < N) ? staged(2, j) : 0.f;
      const float y = in ? staged(3, j) : 0.f;
      const float den = (j == 0) ? b : fmaf(-a, cprev, b);
      if (bad == 0 && bad_pivot(den)) bad = i + 1;
      const float rd = recip(den);
      cp[j] = cc * rd;
      lv[j] = (j == 0) ? a * rd : -a * lprev * rd;
      yv[j] = (j == 0) ? y * rd : fmaf(-a, yprev, y) * rd;
      cprev = cp[j];
      lprev = lv[j];
      yprev = yv[j];
    }
  }
  // ---- upward elimination from row e-1 with t_c = x_e as the right unknown:
  //      x_i = y''_i - l'_i t_{c-1} - r_i t_c  (in place: yv <- y'', lv <- l',
  //      cp <- r).  Row e keeps its downward form (y'_e, l_e, c'_e) for the
  //      reduced system and takes the trivial form x_e = t_c (0, 0, -1).
  const float le = lv[L - 1], ce = cp[L - 1], ye = yv[L - 1];
  yv[L - 1] = 0.f;
  lv[L - 1] = 0.f;
  cp[L - 1] = -1.f;
#pragma unroll
  for (int j = L - 2; j >= 0; --j) {
    const float cj = cp[j];
    yv[j] = fmaf(-cj, yv[j + 1], yv[j]);
    lv[j] = fmaf(-cj, lv[j + 1], lv[j]);
    cp[j] = -cj * cp[j + 1];
  }
  sB[0][c][lane] = lv[0];
  sB[1][c][lane] = cp[0];
  sB[2][c][lane] = yv[0];
  sB[3][c][lane] = le;
  sB[4][c][lane] = ce;
  sB[5][c][lane] = ye;
  __syncthreads();
  if (bad) atomicCAS(&sBad[lane], 0, bad);

  // ---- 2. chunk-end unknowns: P-row tridiagonal system per system, PCR over P lanes
  {
    const int q = threadIdx.x / P;           // system of this lane group (P lanes of a warp)
    const int k = threadIdx.x % P;           // its chunk
    const float le = sB[3][k][q], re = sB[4][k][q], ye = sB[5][k][q];
    const bool last = k == P - 1;
    const float ln = last ? 0.f : sB[0][k + 1][q];
    const float rn = last ? 0.f : sB[1][k + 1][q];
    const float yn = last ? 0.f : sB[2][k + 1][q];
    float sub = k > 0 ? le : 0.f;
    float dia = fmaf(-re, ln, 1.f);
    float sup = last ? 0.f : -re * rn;
    float rhs = fmaf(-re, yn, ye);
#pragma unroll
    for (int d = 1; d < P; d *= 2) {
      const float subm = __shfl_up_sync(0xffffffffu, sub, d, P);
      const float diam = __shfl_up_sync(0xffffffffu, dia, d, P);
      const float supm = __shfl_up_sync(0xffffffffu, sup, d, P);
      const float rhsm = __shfl_up_sync(0xffffffffu, rhs, d, P);
      const float subp = __shfl_down_sync(0xffffffffu, sub, d, P);
      const float diap = __shfl_down_sync(0xffffffffu, dia, d, P);
      const float supp = __shfl_down_sync(0xffffffffu, sup, d, P);
      const float rhsp = __shfl_down_sync(0xffffffffu, rhs, d, P);
      const bool hasm = k >= d, hasp = k + d < P;
      const float al = hasm ? -sub * recip(diam) : 0.f;
      const float be = hasp ? -sup * recip(diap) : 0.f;
      const float nsub = hasm ? al * subm : 0.f;
      const float nsup = hasp ? be * supp : 0.f;
      dia = dia + (hasm ? al * supm : 0.f) + (hasp ? be * subp : 0.f);
      rhs = rhs + (hasm ? al * rhsm : 0.f) + (hasp ? be * rhsp : 0.f);
      sub = nsub;
      sup = nsup;
    }
    if (bad_pivot(dia)) atomicCAS(&sBad[q], 0, min(N, (k + 1) * L));
    sT[k][q] = rhs * recip(dia);
  }
  __syncthreads();

  // ---- 3. every row from t_{c-1} and t_c
  const float tprev = c > 0 ? sT[c - 1][lane] : 0.f;
  const float tcur = sT[c][lane];
#pragma unroll
  for (int j = 0; j < L; ++j) {
    const int i = row0 + j;
    const float x = yv[j] - lv[j] * tprev - cp[j] * tcur;
    if (act && i < N) X[(size_t)i * ld + sb] = x;
  }
  if (c == 0 && act && info) info[s] = sBad[lane];
}

template <typename T>
cudaError_t launch_thread(const void* a, const void* b, const void* c, void* X, int N, int batch, int bs,
                          void* work, int* info, cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  k_tri_thread<T><<<grid, kThreads, 0, st>>>(static_cast<const T*>(a), static_cast<const T*>(b),
                                             static_cast<const T*>(c), static_cast<T*>(X),
                                             static_cast<T*>(work), N, batch, bs, info);
  note_launch();
  return cudaGetLastError();
}

template <int L, int P>
cudaError_t launch_split(const void* a, const void* b, const void* c, void* X, int N, int batch, int bs,
                         int* info, cudaStream_t st) {
  const int grid = (batch + kTriSB - 1) / kTriSB;
  // TMA boxes of BR rows (even, <= 256) covering RS >= N rows
  const int BR = N <= 256 ? ((N + 1) & ~1) : 256;
  const int RS = (N + BR - 1) / BR * BR;
  TriMaps maps;
  const void* ptr[4] = {a, b, c, X};
  // a CTA's 16 systems must lie in one block of a block-interleaved array
  bool tma_ok = bs == 0 || bs % kTriSB == 0;
  for (int k = 0; k < 4 && tma_ok; ++k)
    tma_ok = bs ? tma::encode_3d_blocked(&maps.m[k], ptr[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sizeof(float),
                                         bs, N, batch / bs, kTriSB, (unsigned)BR)
                : tma::encode_2d(&maps.m[k], ptr[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sizeof(float), batch,
                                 N, kTriSB, (unsigned)BR);
  const size_t smem = tma_ok ? (size_t)4 * RS * kTriSB * sizeof(float)
                             : (size_t)4 * L * kTriSB * P * sizeof(float);
  auto kern = tma_ok ? k_tri_split<L, P, true> : k_tri_split<L, P, false>;
  const cudaError_t e = kernel_prepare((const void*)kern, smem, kTriSB * P, nullptr);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTriSB * P, smem, st>>>(maps, static_cast<const float*>(a), static_cast<const float*>(b),
                                          static_cast<const float*>(c), static_cast<float*>(X), N,
                                          batch, bs, RS, BR, info);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

// rows per chunk of the partitioned kernel (at N = 256, batch 262144, 16-row chunks
// run 3 CTAs of 256 threads per SM in 0.212 ms, 8-row chunks 2 CTAs of 512 threads in
// 0.261 ms: fewer reduced-system steps per row, and more CTAs to overlap one tile's
// load with the others' arithmetic)
constexpr int kTriL = 16;

int tri_split_chunks(int N) {
  const int need = (N + kTriL - 1) / kTriL;
  int P = 2;
  while (P < need) P *= 2;
  return P <= 32 ? P : 0;
}

size_t tri_work_bytes(int N, int batch, pent_dtype dt) {
  const size_t elem = dt == PENT_F64 ? sizeof(double) : sizeof(float);
  return (size_t)N * (size_t)batch * elem;
}

cudaError_t tri_solve_batch_df(const void* a, const void* b, const void* c, void* X, int N, int batch, int bs,
                               void* work, int* info, cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  k_tri_thread_df<<<grid, kThreads, 0, st>>>(static_cast<const double*>(a), static_cast<const double*>(b),
                                             static_cast<const double*>(c), static_cast<double*>(X),
                                             static_cast<float2*>(work), N, batch, bs, info);
  note_launch();
  return cudaGetLastError();
}

cudaError_t tri_solve_batch(const void* a, const void* b, const void* c, void* X, int N, int batch, int bs,
                            pent_dtype dt, bool split, void* work, int* info, cudaStream_t st) {
  if (split) {
    switch (tri_split_chunks(N)) {
      case 2: return launch_split<kTriL, 2>(a, b, c, X, N, batch, bs, info, st);
      case 4: return launch_split<kTriL, 4>(a, b, c, X, N, batch, bs, info, st);
      case 8: return launch_split<kTriL, 8>(a, b, c, X, N, batch, bs, info, st);
      case 16: return launch_split<kTriL, 16>(a, b, c, X, N, batch, bs, info, st);
      case 32: return launch_split<kTriL, 32>(a, b, c, X, N, batch, bs, info, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (dt == PENT_F64) return launch_thread<double>(a, b, c, X, N, batch, bs, work, info, st);
  return launch_thread<float>(a, b, c, X, N, batch, bs, work, info, st);
}

}  // namespace pent

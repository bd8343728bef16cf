// Partitioned (split-within-system) shared-matrix solve in double-float.
//
// Same mathematics as the one-thread-per-system solve (forward substitution
// L g = f and back substitution R x = g of "cuPentBatch – A batched
// pentadiagonal solver for NVIDIA GPUs", interleaved layout, factor once), but
// every system is cut into P chunks of L rows, one thread per chunk, so that
// the whole system lives in registers and HBM sees only the two-array minimum
// (read f once, write x once).  Per chunk (tables: pent_factor_split.cu):
//   1. load the chunk, run the forward and the back substitution locally with
//      zero boundary values -> x' (registers); publish the local end values
//      e_c of g;
//   2. boundary states: s_c (the g entering the chunk) and t_c (the x leaving
//      it).  With T > 0 every chunk forms them itself from the T nearest
//      chunks (s_c = sum_k A_{c,k} e_{c-k}, then t_c = sum_k B_{c,k} w_{c+1+k}
//      with w_c = x'_start(c) + Mst_c s_c); the plan chose T so that the
//      couplings dropped are below 2^-64.  With T = 0 one thread per system
//      scans the chunks in order (exact for any matrix);
//   3. x = x' + M1 s0 + M2 s1 + K1 t0 + K2 t1, joined to fp64 and stored.
// Cyclic plans carry Navon's bordering (eqs. (8)–(12)): x_t = S^{-1}(f_t -
// H^T y) from y at rows 0, 1, M-2, M-1, and step 3 subtracts u0 x_t0 + u1 x_t1.
//
// Time steps fused into the same kernel (periodic plans):
//   Cahn–Hilliard (eq. (2)): the load phase builds the right-hand side
//     C_i + k2 (u_{i-1} - 2 u_i + u_{i+1}), u = C^3 - C, from C_{i-1..i+1};
//   Crank–Nicolson (eqs. (5)–(6)): with A = I + sigma_x D4 the step
//     A C' = (2I - A) C equals C' = 2 A^{-1} C - C, so the kernel solves with
//     f = C and stores 2y - C, re-reading its own C_i (still in L2) at the
//     store.
//
// Range: each system is scaled by the power of two that puts its largest
// entry in [1, 2) (an exact operation folded into the integer fp64 <-> pair
// conversions; the Cahn–Hilliard cubic then carries the factor 2^(2s)), so the
// pairs' float exponent range never limits the fp64 contract.  Systems whose
// largest entry is zero, subnormal, non-finite or outside the window of the
// scaled path are solved natively in fp64 by one thread, from their untouched
// input (every store of a block comes after its last load).
//
// Warp layout: 8 consecutive systems x 4 chunks per warp, so every load or
// store instruction moves four 64-byte runs of one row each (whole sectors).
// The per-row tables sit in shared memory with one float4 of padding per
// chunk, so the four chunks a warp reads fall in different banks.  A CTA holds
// SB systems x P chunks; the grid is persistent.
#include "cp_async.cuh"
#include "df64.cuh"
#include "fg.cuh"
#include "pent_internal.cuh"
#include "pent_native.cuh"

namespace pent {
namespace {

using df::D2;

// y += A x for a row-major 2x2 A
__device__ __forceinline__ void mv2(const double* A, double x0, double x1, double& y0, double& y1) {
  y0 = fma(A[0], x0, fma(A[1], x1, y0));
  y1 = fma(A[2], x0, fma(A[3], x1, y1));
}

// y += A x for a row-major 2x2 A of double-float pairs
__device__ __forceinline__ void mv2d(const float2* A, D2 x0, D2 x1, D2& y0, D2& y1) {
  y0 = df::sum3(y0, D2{A[0].x, A[0].y}, x0, D2{A[1].x, A[1].y}, x1);
  y1 = df::sum3(y1, D2{A[2].x, A[2].y}, x0, D2{A[3].x, A[3].y}, x1);
}

// u = q c^3 - c (Cahn–Hilliard chemical potential without the gradient term) for
// c = C 2^-s: the scaled u = (C^3 - C) 2^-s needs q = 2^(2s), an exact power of two
__device__ __forceinline__ D2 cubic_minus(D2 c, float q) {
  const D2 c3 = df::mul(df::mul(c, c), c);
  return df::add(D2{c3.h * q, c3.l * q}, df::neg(c));
}

using fg::kEMin;
using fg::kEMax;
using fg::kEMaxCH;
using fg::cubic_scale;
using fg::pow2_neg;
using fg::pow2_pos;

// rhs_i = C_i + k2 (u_{i-1} - 2 u_i + u_{i+1})   (eq. (2), D2 = [1, -2, 1]/dx^2, k2 = dt/dx^2)
__device__ __forceinline__ D2 ch_rhs(D2 c, D2 um, D2 u0, D2 up, D2 k2) {
  const D2 lap = df::add(df::add(um, up), D2{-2.f * u0.h, -2.f * u0.l});
  return df::add(c, df::mul(k2, lap));
}

// right-hand side / output kind of one launch
constexpr int kRhsPlain = 0;   // solve A x = f in place
constexpr int kRhsCH = 1;      // one Cahn–Hilliard step
constexpr int kRhsCN = 2;      // one Crank–Nicolson step

template <int L, int SB, int MAXT, bool CYC, int RHS>
__global__ void __launch_bounds__(MAXT, (MAXT <= 256 ? 2 : 1))
    k_split_df(const float4* __restrict__ growtab, const double* __restrict__ gchunk,
               const float2* __restrict__ gchunk_df, const double* __restrict__ gextra,
               double* __restrict__ X, int M, int P, int batch, double k2d, const NativeTabs nt) {
  constexpr bool CH = RHS == kRhsCH;
  constexpr bool CN = RHS == kRhsCN;
  static_assert(RHS == kRhsPlain || CYC, "the fused time steps are periodic");
  constexpr int K4 = CYC ? kSpK : kSpK - 1;   // float4 per row kept in shared memory
  constexpr int CS = L * K4 + 1;              // chunk stride (float4), padded
  constexpr int SG = SB / 8;                  // system groups of 8 per CTA
  extern __shared__ float4 smem4[];
  float4* rtab = smem4;                                              // [P][CS]
  // [P][kSpChunk] chunk tables: fp64 for the exact serial scan (T = 0), (hi, lo)
  // pairs for the parallel one, which runs in double-float on the FP32 pipe
  double* ctab = reinterpret_cast<double*>(rtab + (size_t)P * CS);
  const float2* ctab2 = reinterpret_cast<const float2*>(ctab);
  double* sE = ctab + (size_t)P * kSpChunk;      // [SB][P][2] local forward end values e_c
  double* sW = sE + (size_t)SB * P * 2;          // [SB][P][2] x'_start (serial) or w_c (parallel)
  double* sS = sW + (size_t)SB * P * 2;          // [SB][P][2] s_c (serial scan)
  double* sT = sS + (size_t)SB * P * 2;          // [SB][P][2] t_c (serial scan)
  double* sX = sT + (size_t)SB * P * 2;          // [SB][8]   cyclic: y and x_t
  uint32_t* smax = reinterpret_cast<uint32_t*>(sX + (size_t)SB * 8);   // [SB] largest |entry| bits

  for (int t = threadIdx.x; t < P * L * K4; t += blockDim.x) {
    const int row = t / K4, k = t % K4;
    cp_async16(&rtab[(row / L) * CS + (row % L) * K4 + k], &growtab[(size_t)row * kSpK + k]);
  }
  const int T = (int)gextra[18];
  if (T > 0) {
    for (int t = threadIdx.x; t < P * kSpChunk / 2; t += blockDim.x)
      cp_async16(&ctab[2 * t], &gchunk_df[2 * t]);
  } else {
    for (int t = threadIdx.x; t < P * kSpChunk / 2; t += blockDim.x) cp_async16(&ctab[2 * t], &gchunk[2 * t]);
  }
  for (int t = threadIdx.x; t < SB; t += blockDim.x) smax[t] = 0u;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int sys = (w % SG) * 8 + (lane & 7);
  const int c = (w / SG) * 4 + (lane >> 3);
  const int row0 = c * L;
  // the first block's rows of this chunk start towards L2 while the tables arrive,
  // so a short solve waits for one memory latency instead of two
  if (blockIdx.x * SB + sys < batch) {
    const double* pf = X + (long long)row0 * batch + blockIdx.x * SB + sys;
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (row0 + j < M) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf + (long long)j * batch));
  }
  cp_async_wait_all();
  __syncthreads();

  const float4* ctb = rtab + (size_t)c * CS;     // this chunk's rows
  const int reach = CYC ? (int)gextra[19] : 0;
  const bool needU = CYC && (c < reach || c > (M - 1) / L - reach);   // x_t correction not negligible
  const float2* ct = ctab2 + (size_t)c * kSpChunk;
  const long long ld = batch;
  const int nblk = (batch + SB - 1) / SB;

  for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int s = blk * SB + sys;
    const bool act = s < batch;
    double* p = X + (long long)row0 * ld + (act ? s : 0);

    // ---- 1. the system's largest entry sets its scale: a first pass over this
    // chunk's rows (and, for the chunk-0 thread of a cyclic plan, the two border
    // rows) takes the maximum, one barrier shares it; the loads below then find
    // the rows in cache.  Then: load, local forward (zero incoming state), local
    // backward.
    // off = (e - 127) << 20 for the system's exponent field e: the rebias of
    // both conversions (f 2^-s in, x 2^s out); e = (off >> 20) + 127
    uint32_t off = 0u;
    bool native = false, keep = false;
    float q = 1.f;
    // The fused time steps load this thread's rows once, before the maximum,
    // and keep them for the right-hand side (Cahn–Hilliard: rows row0-1 ..
    // row0+L, row -1 wrapping to N-1 = M+1, for C_{i-1}, C_i, C_{i+1}): one
    // memory latency per block instead of two (0.267 -> 0.238 ms per
    // Cahn–Hilliard step, 0.0375 -> 0.0355 ms per Crank–Nicolson step).  The
    // plain solve reads its rows twice (the second time from cache): holding
    // them across the barrier spilled registers there (0.031 -> 0.033 ms).  Every
    // load of a block precedes its first store (barriers below).
    constexpr bool EARLY = RHS != kRhsPlain;
    constexpr int NV = CH ? L + 2 : L;
    constexpr int J0 = CH ? 1 : 0;                      // cv[J0 + j] is row row0 + j
    double cv[NV];
    if constexpr (CH) {
#pragma unroll
      for (int j = 0; j < L + 2; ++j) {
        const int i = row0 - 1 + j;
        const int iw = i < 0 ? M + 1 : i;
        cv[j] = (act && i <= M) ? X[(long long)iw * ld + s] : 0.0;
      }
    } else if constexpr (EARLY) {
#pragma unroll
      for (int j = 0; j < L; ++j) cv[j] = (act && row0 + j < M) ? p[j * ld] : 0.0;
    }
    {
      // magnitude word: largest high word, bit 0 set if any low word is nonzero
      uint32_t mx = 0u, nz = 0u;
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (act && row0 + j < M) {
          const double v = EARLY ? cv[J0 + j] : p[j * ld];
          mx = max(mx, fg::mag_bits(v));
          nz |= (uint32_t)__double2loint(v);
        }
      if (CYC && c == 0 && act) {
        const double v0 = X[(long long)M * ld + s], v1 = X[(long long)(M + 1) * ld + s];
        mx = max(mx, fg::mag_pair(v0, v1, nz));
      }
      atomicMax(&smax[sys], mx | (nz != 0u ? 1u : 0u));
      __syncthreads();
      const uint32_t e = smax[sys] >> 20;
      const bool fast = e >= kEMin && e <= (CH ? kEMaxCH : kEMax);
      // an all-zero state is its own result (solve, Crank–Nicolson and
      // Cahn–Hilliard all map 0 to 0, in place): nothing is stored
      keep = smax[sys] == 0u;
      native = act && !fast && !keep;
      off = fg::in_offset(fast ? e : 1023u);
      if constexpr (CH) q = cubic_scale(fast ? e : 1023u);
    }
    const bool store = act && !native && !keep;
    // f * 2^-s as a pair
    auto sdf = [&](double v) {
      float h, lo;
      fg::split(v, off, h, lo);
      return D2{h, lo};
    };
    D2 v[L];
    if constexpr (CH) {
      // right-hand side from C_{i-1}, C_i, C_{i+1}
      const D2 k2 = df::from_double(k2d);
      D2 cc = sdf(cv[1]);
      D2 um = cubic_minus(sdf(cv[0]), q), u0 = cubic_minus(cc, q);
      D2 a1{0.f, 0.f}, a2{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < L; ++j) {
        const D2 cn = sdf(cv[j + 2]);
        const D2 up = cubic_minus(cn, q);
        D2 f = ch_rhs(cc, um, u0, up, k2);
        if (row0 + j >= M) f = D2{0.f, 0.f};
        const float4 c0 = ctb[j * K4];
        const float4 c1 = ctb[j * K4 + 1];
        const D2 g = df::sum3p(D2{c0.x, c0.y}, f, D2{c0.z, c0.w}, a2, D2{c1.x, c1.y}, a1);
        v[j] = g;
        a2 = a1;
        a1 = g;
        um = u0;
        u0 = up;
        cc = cn;
      }
    } else {
      if constexpr (!EARLY) {
#pragma unroll
        for (int j = 0; j < L; ++j) cv[j] = (act && row0 + j < M) ? p[j * ld] : 0.0;
      }
      const double* fv = cv;
      D2 a1{0.f, 0.f}, a2{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < L; ++j) {
        const float4 c0 = ctb[j * K4];
        const float4 c1 = ctb[j * K4 + 1];
        const D2 g = df::sum3p(D2{c0.x, c0.y}, sdf(fv[j]), D2{c0.z, c0.w}, a2,
                               D2{c1.x, c1.y}, a1);
        v[j] = g;
        a2 = a1;
        a1 = g;
      }
    }
    if (T > 0) {
      float2* eo = reinterpret_cast<float2*>(sE) + ((size_t)sys * P + c) * 2;
      eo[0] = make_float2(v[L - 2].h, v[L - 2].l);
      eo[1] = make_float2(v[L - 1].h, v[L - 1].l);
    } else {
      double* eo = sE + ((size_t)sys * P + c) * 2;
      eo[0] = df::to_double(v[L - 2]);
      eo[1] = df::to_double(v[L - 1]);
    }
    {
      D2 a1{0.f, 0.f}, a2{0.f, 0.f};
#pragma unroll
      for (int j = L - 1; j >= 0; --j) {
        const float4 c2 = ctb[j * K4 + 2];
        const D2 y = df::sum3(v[j], D2{c2.x, c2.y}, a1, D2{c2.z, c2.w}, a2);
        v[j] = y;
        a2 = a1;
        a1 = y;
      }
    }
    const D2 xs0 = v[0], xs1 = v[1];   // x'_start(c)
    // x' at rows M-2, M-1 (cyclic): only the owning chunks keep them
    double xm2 = 0.0, xm1 = 0.0;
    if (CYC && row0 <= M - 1 && M - 2 < row0 + L) {
#pragma unroll
      for (int j = 0; j < L; ++j) {
        if (row0 + j == M - 2) xm2 = df::to_double(v[j]);
        if (row0 + j == M - 1) xm1 = df::to_double(v[j]);
      }
    }

    // ---- 2. boundary states s_c (entering) and t_c (leaving): the truncated
    // parallel scan in double-float on the FP32 pipe (in fp64 its few operations
    // per thread queue on the slow fp64 pipe between two barriers, with every warp
    // waiting), the exact serial one (testing, slowly decaying couplings) in fp64
    D2 S0{0.f, 0.f}, S1{0.f, 0.f}, T0{0.f, 0.f}, T1{0.f, 0.f};
    double* xc = sX + (size_t)sys * 8;
    if (T > 0) {
      __syncthreads();                                   // e_c published, smax read
      if (c == 0) smax[sys] = 0u;                        // next block (ordered by the next barrier)
      const float2* E = reinterpret_cast<const float2*>(sE) + (size_t)sys * P * 2;
      for (int k = 1; k <= T && k <= c; ++k) {           // s_c = sum_k A_{c,k} e_{c-k}
        const D2 ea{E[2 * (c - k)].x, E[2 * (c - k)].y}, eb{E[2 * (c - k) + 1].x, E[2 * (c - k) + 1].y};
        if (k == 1) { S0 = df::add(S0, ea); S1 = df::add(S1, eb); }
        else mv2d(ct + 12 + 4 * (k - 2), ea, eb, S0, S1);
      }
      D2 w0 = xs0, w1 = xs1;
      mv2d(ct + 4, S0, S1, w0, w1);                      // w_c = x'_start + Mst_c s_c
      float2* wo = reinterpret_cast<float2*>(sW) + ((size_t)sys * P + c) * 2;
      wo[0] = make_float2(w0.h, w0.l);
      wo[1] = make_float2(w1.h, w1.l);
      __syncthreads();                                   // w_c published
      const float2* Wv = reinterpret_cast<const float2*>(sW) + (size_t)sys * P * 2;
      for (int k = 0; k < T && c + 1 + k < P; ++k) {     // t_c = sum_k B_{c,k} w_{c+1+k}
        const D2 wa{Wv[2 * (c + 1 + k)].x, Wv[2 * (c + 1 + k)].y};
        const D2 wb{Wv[2 * (c + 1 + k) + 1].x, Wv[2 * (c + 1 + k) + 1].y};
        if (k == 0) { T0 = df::add(T0, wa); T1 = df::add(T1, wb); }
        else mv2d(ct + 24 + 4 * (k - 1), wa, wb, T0, T1);
      }
      if (CYC) {
        if (c == 0) {                                    // y at rows 0, 1
          D2 y0 = w0, y1 = w1;
          mv2d(ct + 8, T0, T1, y0, y1);
          xc[2] = df::to_double(y0);
          xc[3] = df::to_double(y1);
        }
        if (row0 <= M - 1 && M - 2 < row0 + L) {
          const double s0 = df::to_double(S0), s1 = df::to_double(S1);
          const double t0 = df::to_double(T0), t1 = df::to_double(T1);
          if (row0 <= M - 2 && M - 2 < row0 + L)
            xc[0] = xm2 + gextra[10] * s0 + gextra[11] * s1 + gextra[14] * t0 + gextra[15] * t1;
          if (row0 <= M - 1 && M - 1 < row0 + L)
            xc[1] = xm1 + gextra[12] * s0 + gextra[13] * s1 + gextra[16] * t0 + gextra[17] * t1;
        }
      }
    } else {
      double* wo = sW + ((size_t)sys * P + c) * 2;
      wo[0] = df::to_double(xs0);
      wo[1] = df::to_double(xs1);
      if (CYC) {
        if (row0 <= M - 2 && M - 2 < row0 + L) xc[0] = xm2;
        if (row0 <= M - 1 && M - 1 < row0 + L) xc[1] = xm1;
      }
      __syncthreads();                                   // e_c, x'_start published, smax read
      if (c == 0) smax[sys] = 0u;                        // next block (ordered by the next barrier)
      if (c == 0) {                                      // exact serial scan, one thread per system
        const double* E = sE + (size_t)sys * P * 2;
        const double* Wv = sW + (size_t)sys * P * 2;
        double* S = sS + (size_t)sys * P * 2;
        double* Tt = sT + (size_t)sys * P * 2;
        double a0 = 0.0, a1 = 0.0;
        for (int k = 0; k < P; ++k) {                    // s_{k+1} = e_k + Phi_k s_k
          S[2 * k] = a0;
          S[2 * k + 1] = a1;
          double n0 = E[2 * k], n1 = E[2 * k + 1];
          mv2(ctab + (size_t)k * kSpChunk, a0, a1, n0, n1);
          a0 = n0;
          a1 = n1;
        }
        double b0 = 0.0, b1 = 0.0;
        for (int k = P - 1; k >= 0; --k) {               // x at the start of chunk k
          Tt[2 * k] = b0;
          Tt[2 * k + 1] = b1;
          const double* ck = ctab + (size_t)k * kSpChunk;
          double x0 = Wv[2 * k], x1 = Wv[2 * k + 1];
          mv2(ck + 4, S[2 * k], S[2 * k + 1], x0, x1);
          mv2(ck + 8, b0, b1, x0, x1);
          b0 = x0;
          b1 = x1;
        }
        if (CYC) {
          const int k2 = (M - 2) / L, k1 = (M - 1) / L;
          xc[0] += gextra[10] * S[2 * k2] + gextra[11] * S[2 * k2 + 1] + gextra[14] * Tt[2 * k2] +
                   gextra[15] * Tt[2 * k2 + 1];
          xc[1] += gextra[12] * S[2 * k1] + gextra[13] * S[2 * k1 + 1] + gextra[16] * Tt[2 * k1] +
                   gextra[17] * Tt[2 * k1 + 1];
          xc[2] = b0;
          xc[3] = b1;
        }
      }
      __syncthreads();
      S0 = df::from_double(sS[((size_t)sys * P + c) * 2]);
      S1 = df::from_double(sS[((size_t)sys * P + c) * 2 + 1]);
      T0 = df::from_double(sT[((size_t)sys * P + c) * 2]);
      T1 = df::from_double(sT[((size_t)sys * P + c) * 2 + 1]);
    }
    // cyclic: x_t = S^{-1}(f_t - H^T y)   (eq. (12))
    double xt0 = 0.0, xt1 = 0.0;
    if (CYC) {
      __syncthreads();                                   // y published
      if (c == 0) {
        const double r0 = gextra[4] * xc[0] + gextra[5] * xc[1] + gextra[6] * xc[2];
        const double r1 = gextra[7] * xc[1] + gextra[8] * xc[2] + gextra[9] * xc[3];
        // the border rows in the system's scale (all doubles here are scaled)
        double ft0 = 0.0, ft1 = 0.0;
        if (act) {
          if constexpr (CH) {
            // tail rows N-2 = M and N-1 = M+1 need C at M-1, M, M+1 and 0
            const D2 k2 = df::from_double(k2d);
            const D2 cA = sdf(X[(long long)(M - 1) * ld + s]);
            const D2 cB = sdf(X[(long long)M * ld + s]);
            const D2 cC = sdf(X[(long long)(M + 1) * ld + s]);
            const D2 cD = sdf(X[s]);
            const D2 uA = cubic_minus(cA, q), uB = cubic_minus(cB, q), uC = cubic_minus(cC, q);
            const D2 uD = cubic_minus(cD, q);
            ft0 = df::to_double(ch_rhs(cB, uA, uB, uC, k2));
            ft1 = df::to_double(ch_rhs(cC, uB, uC, uD, k2));
          } else {
            ft0 = X[(long long)M * ld + s] * pow2_neg((off >> 20) + 127u);
            ft1 = X[(long long)(M + 1) * ld + s] * pow2_neg((off >> 20) + 127u);
          }
        }
        const double u0 = gextra[0] * (ft0 - r0) + gextra[1] * (ft1 - r1);
        const double u1 = gextra[2] * (ft0 - r0) + gextra[3] * (ft1 - r1);
        xc[4] = u0;
        xc[5] = u1;
        if (store) {
          X[(long long)M * ld + s] = (CN ? 2.0 * u0 - ft0 : u0) * pow2_pos((off >> 20) + 127u);
          X[(long long)(M + 1) * ld + s] = (CN ? 2.0 * u1 - ft1 : u1) * pow2_pos((off >> 20) + 127u);
        }
      }
      __syncthreads();
      xt0 = xc[4];
      xt1 = xc[5];
    }

    // ---- 3. x = x' + M1 s0 + M2 s1 + K1 t0 + K2 t1 (- u0 x_t0 - u1 x_t1), store
    {
      const D2 X0 = df::from_double(-xt0), X1 = df::from_double(-xt1);
      if (CYC && needU) {
#pragma unroll
        for (int j = 0; j < L; ++j) {
          const float4 c1 = ctb[j * K4 + 1], c5 = ctb[j * K4 + 5];
          const D2 x = df::axpy(v[j], D2{c1.z, c1.w}, X0);
          v[j] = df::axpy(x, D2{c5.x, c5.y}, X1);
        }
      }
      constexpr int G = CN ? 8 : L;                    // rows per group (CN re-reads C)
#pragma unroll
      for (int j0 = 0; j0 < L; j0 += G) {
        double cold[CN ? G : 1];
        if constexpr (CN) {
#pragma unroll
          for (int u = 0; u < G; ++u) cold[u] = (act && row0 + j0 + u < M) ? p[(j0 + u) * ld] : 0.0;
        }
#pragma unroll
        for (int u = 0; u < G; ++u) {
          const int j = j0 + u;
          const float4 c3 = ctb[j * K4 + 3], c4 = ctb[j * K4 + 4];
          D2 x = df::axpy(v[j], D2{c3.x, c3.y}, S0);
          x = df::axpy(x, D2{c3.z, c3.w}, S1);
          x = df::axpy(x, D2{c4.x, c4.y}, T0);
          x = df::axpy(x, D2{c4.z, c4.w}, T1);
          if constexpr (CN) x = df::add(D2{2.f * x.h, 2.f * x.l}, df::neg(sdf(cold[u])));
          // three rows in four join through integers, off the slow fp64 pipe
          const double xo = (j & 3) != 0 ? fg::join_int(x.h, x.l, off) : fg::join(x.h, x.l, off);
          fg::store_cs_if(p + j * ld, xo, store && row0 + j < M);
        }
      }
    }
    // systems outside the scaled path: one thread solves the column in fp64 from
    // its untouched input (cyclic plans: N = M + 2 rows)
    if (native && c == 0) {
      if constexpr (CH) native_ch_col(nt, X + s, M + 2, (size_t)ld, k2d, 1);
      else if constexpr (CN) native_cn_col(nt, X + s, M + 2, (size_t)ld, 1);
      else native_solve_col(nt, X + s, M, (size_t)ld, CYC ? 1 : 0);
    }
  }
}

template <int L, int SB, int MAXT, bool CYC, int RHS = kRhsPlain>
cudaError_t launch(const pent_plan_s& p, double* X, int batch, cudaStream_t st, double k2 = 0.0) {
  const int P = p.sp_P;
  const size_t smem = split_smem_bytes(L, P, SB, CYC);
  auto kern = k_split_df<L, SB, MAXT, CYC, RHS>;
  const int nblk = (batch + SB - 1) / SB;
  // persistent grid: as many CTAs as fit on every SM at once (registers and
  // shared memory of this instance), capped by the number of system blocks
  int per_sm = 0;
  const cudaError_t e = kernel_prepare((const void*)kern, smem, SB * P, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  int grid = p.df_ctas > 0 ? p.df_ctas : per_sm * p.num_sms;
  if (grid > nblk) grid = nblk;
  const NativeTabs nt{p.coef64, p.tail64, p.bands};
  kern<<<grid, SB * P, smem, st>>>(p.sptab, p.spchunk, p.spchunk_df, p.spextra, X, p.M, P, batch, k2, nt);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

size_t split_smem_bytes(int L, int P, int SB, int cyclic) {
  const int K4 = cyclic ? kSpK : kSpK - 1;
  return (size_t)P * (L * K4 + 1) * sizeof(float4) +
         ((size_t)P * kSpChunk + 4 * (size_t)SB * P * 2 + (size_t)SB * 8) * sizeof(double) +
         (size_t)SB * sizeof(uint32_t);
}

// Cyclic plans with L = 32 and P <= 32 run 16 systems per CTA (one copy of the
// tables in shared memory serves more systems) unless the batch is too small
// to give every SM one such CTA; then 8, for twice as many CTAs.
template <int RHS>
cudaError_t launch_cyclic(const pent_plan_s& p, double* X, int batch, cudaStream_t st, double k2) {
  if (p.sp_L == 16) return launch<16, 8, 512, true, RHS>(p, X, batch, st, k2);
  const bool wide = p.sp_P <= 32 && batch > 16 * p.num_sms;
  return wide ? launch<32, 16, 512, true, RHS>(p, X, batch, st, k2)
              : launch<32, 8, 512, true, RHS>(p, X, batch, st, k2);
}

cudaError_t shared_split_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  // p.sp_L and p.sp_P were fixed at plan time (P % 4 == 0, SB * P threads)
  if (p.cyclic) return launch_cyclic<kRhsPlain>(p, X, batch, st, 0.0);
  if (p.sp_L == 16) return launch<16, 8, 512, false>(p, X, batch, st);
  return p.sp_P <= 32 ? launch<32, 8, 256, false>(p, X, batch, st)
                      : launch<32, 8, 512, false>(p, X, batch, st);
}

cudaError_t ch_split_df(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st) {
  return launch_cyclic<kRhsCH>(p, X, batch, st, k2);
}

cudaError_t cn_split_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  return launch_cyclic<kRhsCN>(p, X, batch, st, 0.0);
}

}  // namespace pent

// Shared-matrix batched solve in double-float arithmetic: twisted sweeps,
// SPT adjacent systems per thread.
//
// Mathematics: forward substitution L g = f and back substitution R x = g of
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs" (factor once,
// interleaved layout), with the elimination order of the twisted factorisation
// (pent_factor_twisted.cu): warps of the "top" half sweep rows 0..m-1 downwards,
// warps of the "bottom" half sweep rows M-1..m upwards with the factors of the
// reversed block, the two meet in a 4x4 system in x_{m-2..m+1}, then both
// back-substitute outwards.  Cyclic plans carry Navon's bordering (eqs.
// (8)–(12)) in the same pass (q . f accumulated inwards, u x_t subtracted
// outwards).
//
// GB300 plan:
//  * double-float arithmetic on the FP32 pipe (df64.cuh); fp64 hardware only
//    for the hi+lo join of each output and the 4x4 meeting system;
//  * SPT adjacent systems per thread: one 8*SPT-byte access per row, and the
//    shared coefficient loads and address arithmetic serve SPT systems;
//  * persistent CTAs over blocks of SPB systems: the number of systems in
//    flight, hence the L2 footprint of the in-place intermediate g, is
//    bounded by the grid size; g (a float pair) overwrites f in place and is
//    read back by the outward sweep, mostly from L2;
//  * register ring of two blocks of kU rows, loads issued one block ahead;
//    full blocks run without per-row guards, a ragged last block with them.
#include <type_traits>

#include "cp_async.cuh"
#include "df64.cuh"
#include "pent_internal.cuh"

namespace pent {
namespace {

using df::D2;

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- SPT-wide memory accesses (addresses 8*SPT-byte aligned) -------------
template <int SPT>
__device__ __forceinline__ void ld_f(const char* p, double* v) {
  if constexpr (SPT == 2) {
    const double2 t = *reinterpret_cast<const double2*>(p);
    v[0] = t.x;
    v[1] = t.y;
  } else {
    v[0] = *reinterpret_cast<const double*>(p);
  }
}
template <int SPT>
__device__ __forceinline__ void st_g(char* p, const D2* g) {
  if constexpr (SPT == 2)
    *reinterpret_cast<float4*>(p) = make_float4(g[0].h, g[0].l, g[1].h, g[1].l);
  else
    *reinterpret_cast<float2*>(p) = make_float2(g[0].h, g[0].l);
}
template <int SPT>
__device__ __forceinline__ void ld_g(const char* p, D2* g) {
  if constexpr (SPT == 2) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    g[0] = D2{t.x, t.y};
    g[1] = D2{t.z, t.w};
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    g[0] = D2{t.x, t.y};
  }
}
template <int SPT>
__device__ __forceinline__ void st_x(char* p, const double* x) {
  if constexpr (SPT == 2)
    __stcs(reinterpret_cast<double2*>(p), make_double2(x[0], x[1]));
  else
    __stcs(reinterpret_cast<double*>(p), x[0]);
}

// One thread's state for SPT systems.
template <int SPT>
struct Lane {
  D2 a1[SPT], a2[SPT];     // recurrence state: value at j-1 and j-2 (local order)
  D2 acc0[SPT], acc1[SPT]; // cyclic dot products q_k . f
};

// inward row: g = r f + P g_{j-2} + Q g_{j-1}; returns g in s.a1 (shifts state)
template <int SPT, bool CYC>
__device__ __forceinline__ void inward_row(const float4* __restrict__ row, const double* f,
                                           Lane<SPT>& s, D2* g) {
  const float4 c0 = row[0], c1 = row[1];
  float4 c2, c3;
  if (CYC) { c2 = row[2]; c3 = row[3]; }
#pragma unroll
  for (int t = 0; t < SPT; ++t) {
    const D2 fv = df::from_double(f[t]);
    g[t] = df::sum3p(D2{c0.x, c0.y}, fv, D2{c0.z, c0.w}, s.a2[t], D2{c1.x, c1.y}, s.a1[t]);
    if (CYC) {
      s.acc0[t] = df::axpy(s.acc0[t], D2{c2.z, c2.w}, fv);
      s.acc1[t] = df::axpy(s.acc1[t], D2{c3.x, c3.y}, fv);
    }
    s.a2[t] = s.a1[t];
    s.a1[t] = g[t];
  }
}

// outward row: y = g + C y_{j+1} + D y_{j+2}; x = y (- u0 x_t0 - u1 x_t1 if cyclic)
template <int SPT, bool CYC>
__device__ __forceinline__ void outward_row(const float4* __restrict__ row, const D2* g,
                                            Lane<SPT>& s, const D2* nx0, const D2* nx1,
                                            double* x) {
  const float4 c1 = row[1], c2 = row[2];
  float4 c3, c4;
  if (CYC) { c3 = row[3]; c4 = row[4]; }
#pragma unroll
  for (int t = 0; t < SPT; ++t) {
    const D2 y = df::sum3(g[t], D2{c1.z, c1.w}, s.a1[t], D2{c2.x, c2.y}, s.a2[t]);
    D2 xv = y;
    if (CYC) xv = df::axpy(df::axpy(xv, D2{c3.z, c3.w}, nx0[t]), D2{c4.x, c4.y}, nx1[t]);
    x[t] = df::to_double(xv);
    s.a2[t] = s.a1[t];
    s.a1[t] = y;
  }
}

// SPB systems per CTA, SPT per thread, KU rows per prefetch block.
template <int SPT, int SPB, int KU, bool CYC>
__global__ void __launch_bounds__(2 * SPB / SPT)
    k_twisted_df(const float4* __restrict__ gtab, const double* __restrict__ twist,
                 double* __restrict__ X, int M, int m, int batch) {
  constexpr int TPD = SPB / SPT;   // threads per direction
  constexpr int NX = CYC ? 8 : 4;
  extern __shared__ float4 stab[];
  __shared__ double sx[TPD][SPT][NX];
  __shared__ double sT[kTwistCount];
  for (int t = threadIdx.x; t < M * kTwK; t += blockDim.x) cp_async16(&stab[t], &gtab[t]);
  cp_async_wait_all();
  if (threadIdx.x < kTwistCount) sT[threadIdx.x] = twist[threadIdx.x];
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool top = warp < TPD / 32;
  const int grp = top ? warp : warp - TPD / 32;
  const int tl = grp * 32 + lane;
  const float4* tab = stab + (top ? 0 : m * kTwK);
  const int rows = top ? m : M - m;
  const long long ld = batch;
  const long long stepB = (top ? ld : -ld) * (long long)sizeof(double);
  const int nblk = (batch + SPB - 1) / SPB;
  const int nb_in = (rows + KU - 1) / KU;
  const int jtop = rows - 3;                      // first outward row (local)
  const int nb_out = (jtop + 1 + KU - 1) / KU;

  for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int s0 = blk * SPB + tl * SPT;
    const bool act = s0 < batch;
    // inactive lanes read system 0 (harmless) and never store
    char* p0 = reinterpret_cast<char*>(X + (top ? 0 : (long long)(M - 1) * ld) + (act ? s0 : 0));
    Lane<SPT> st;
#pragma unroll
    for (int t = 0; t < SPT; ++t) {
      st.a1[t] = st.a2[t] = st.acc0[t] = st.acc1[t] = D2{0.f, 0.f};
    }

    // ------------------------------------------------ inward sweep
    double fa[KU][SPT], fb[KU][SPT];
    auto load_in = [&](double (*buf)[SPT], int b) {
      const int j0 = b * KU;
      const char* q = p0 + (long long)j0 * stepB;
      if (j0 + KU <= rows) {
#pragma unroll
        for (int u = 0; u < KU; ++u) { ld_f<SPT>(q, buf[u]); q += stepB; }
      } else if (j0 < rows) {
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          if (j0 + u < rows) ld_f<SPT>(q, buf[u]);
          q += stepB;
        }
      }
    };
    auto run_in = [&](double (*buf)[SPT], int b) {
      const int j0 = b * KU;
      char* q = p0 + (long long)j0 * stepB;
      const float4* row = tab + j0 * kTwK;
      D2 g[SPT];
      if (j0 + KU <= rows) {
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          inward_row<SPT, CYC>(row + u * kTwK, buf[u], st, g);
          if (act) st_g<SPT>(q, g);
          q += stepB;
        }
      } else {
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          if (j0 + u < rows) {
            inward_row<SPT, CYC>(row + u * kTwK, buf[u], st, g);
            if (act) st_g<SPT>(q, g);
          }
          q += stepB;
        }
      }
    };
    load_in(fa, 0);
    load_in(fb, 1);
    for (int b = 0; b < nb_in; b += 2) {
      run_in(fa, b);
      load_in(fa, b + 2);
      if (b + 1 < nb_in) {
        run_in(fb, b + 1);
        load_in(fb, b + 3);
      }
    }

    // ------------------------------------------------ meeting point (fp64)
    // top: a2 = g_{m-2}, a1 = g_{m-1}; bottom: a1 = g~ at row m, a2 = g~ at row m+1.
#pragma unroll
    for (int t = 0; t < SPT; ++t) {
      if (top) {
        sx[tl][t][0] = df::to_double(st.a2[t]);
        sx[tl][t][1] = df::to_double(st.a1[t]);
        if (CYC) { sx[tl][t][4] = df::to_double(st.acc0[t]); sx[tl][t][5] = df::to_double(st.acc1[t]); }
      } else {
        sx[tl][t][2] = df::to_double(st.a1[t]);
        sx[tl][t][3] = df::to_double(st.a2[t]);
        if (CYC) { sx[tl][t][6] = df::to_double(st.acc0[t]); sx[tl][t][7] = df::to_double(st.acc1[t]); }
      }
    }
    named_barrier(1 + grp, 64);
    const double* Ti = sT + (top ? 0 : 8);   // my two rows of T^{-1}
    double v0[SPT], v1[SPT];
    D2 nx0[SPT], nx1[SPT];
    double xt0[SPT], xt1[SPT];
#pragma unroll
    for (int t = 0; t < SPT; ++t) {
      const double w0 = sx[tl][t][0], w1 = sx[tl][t][1], w2 = sx[tl][t][2], w3 = sx[tl][t][3];
      v0[t] = Ti[0] * w0 + Ti[1] * w1 + Ti[2] * w2 + Ti[3] * w3;
      v1[t] = Ti[4] * w0 + Ti[5] * w1 + Ti[6] * w2 + Ti[7] * w3;
      nx0[t] = nx1[t] = D2{0.f, 0.f};
    }
    if (CYC) {
      double ft0[SPT], ft1[SPT];
      const char* pt = reinterpret_cast<const char*>(X + (long long)M * ld + (act ? s0 : 0));
      ld_f<SPT>(pt, ft0);
      ld_f<SPT>(pt + ld * (long long)sizeof(double), ft1);
#pragma unroll
      for (int t = 0; t < SPT; ++t) {
        const double r0 = ft0[t] - (sx[tl][t][4] + sx[tl][t][6]);
        const double r1 = ft1[t] - (sx[tl][t][5] + sx[tl][t][7]);
        xt0[t] = sT[16] * r0 + sT[17] * r1;
        xt1[t] = sT[18] * r0 + sT[19] * r1;
        nx0[t] = df::from_double(-xt0[t]);
        nx1[t] = df::from_double(-xt1[t]);
      }
    }
    named_barrier(1 + grp, 64);   // partner has read sx (and f_t) before reuse / overwrite
    if (CYC && act && !top) {
      char* pt = reinterpret_cast<char*>(X + (long long)M * ld + s0);
      st_x<SPT>(pt, xt0);
      st_x<SPT>(pt + ld * (long long)sizeof(double), xt1);
    }
    // meeting rows: top local m-2 <- v0, m-1 <- v1; bottom local Mb-1 (row m) <- v0,
    // Mb-2 (row m+1) <- v1.  Outward state: a1 = value at j+1, a2 = at j+2.
    {
      const int jA = top ? rows - 2 : rows - 1;
      const int jB = top ? rows - 1 : rows - 2;
      double xa[SPT], xb[SPT];
#pragma unroll
      for (int t = 0; t < SPT; ++t) {
        const D2 a = df::from_double(v0[t]), b = df::from_double(v1[t]);
        st.a1[t] = top ? a : b;
        st.a2[t] = top ? b : a;
        D2 ya = a, yb = b;
        if (CYC) {
          const float4 cA3 = tab[jA * kTwK + 3], cA4 = tab[jA * kTwK + 4];
          const float4 cB3 = tab[jB * kTwK + 3], cB4 = tab[jB * kTwK + 4];
          ya = df::axpy(df::axpy(ya, D2{cA3.z, cA3.w}, nx0[t]), D2{cA4.x, cA4.y}, nx1[t]);
          yb = df::axpy(df::axpy(yb, D2{cB3.z, cB3.w}, nx0[t]), D2{cB4.x, cB4.y}, nx1[t]);
          xa[t] = df::to_double(ya);
          xb[t] = df::to_double(yb);
        } else {
          xa[t] = v0[t];
          xb[t] = v1[t];
        }
      }
      if (act) {
        st_x<SPT>(p0 + (long long)jA * stepB, xa);
        st_x<SPT>(p0 + (long long)jB * stepB, xb);
      }
    }

    // ------------------------------------------------ outward sweep, local rows jtop..0
    D2 ga[KU][SPT], gb[KU][SPT];
    auto load_out = [&](D2 (*buf)[SPT], int b) {
      const int j0 = jtop - b * KU;
      const char* q = p0 + (long long)j0 * stepB;
      if (j0 - (KU - 1) >= 0) {
#pragma unroll
        for (int u = 0; u < KU; ++u) { ld_g<SPT>(q, buf[u]); q -= stepB; }
      } else if (j0 >= 0) {
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          if (j0 - u >= 0) ld_g<SPT>(q, buf[u]);
          q -= stepB;
        }
      }
    };
    auto run_out = [&](D2 (*buf)[SPT], int b) {
      const int j0 = jtop - b * KU;
      char* q = p0 + (long long)j0 * stepB;
      const float4* row = tab + j0 * kTwK;
      double x[SPT];
      if (j0 - (KU - 1) >= 0) {
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          outward_row<SPT, CYC>(row - u * kTwK, buf[u], st, nx0, nx1, x);
          if (act) st_x<SPT>(q, x);
          q -= stepB;
        }
      } else {
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          if (j0 - u >= 0) {
            outward_row<SPT, CYC>(row - u * kTwK, buf[u], st, nx0, nx1, x);
            if (act) st_x<SPT>(q, x);
          }
          q -= stepB;
        }
      }
    };
    load_out(ga, 0);
    load_out(gb, 1);
    for (int b = 0; b < nb_out; b += 2) {
      run_out(ga, b);
      load_out(ga, b + 2);
      if (b + 1 < nb_out) {
        run_out(gb, b + 1);
        load_out(gb, b + 3);
      }
    }
  }
}

// ---- asynchronous row streaming (cp.async: global -> shared, no registers held;
// the copy helpers are in cp_async.cuh)
__device__ __forceinline__ void unpack2(const uint4 r, double* v) {
  v[0] = __hiloint2double((int)r.y, (int)r.x);
  v[1] = __hiloint2double((int)r.w, (int)r.z);
}

// Same sweeps as k_twisted_df with two systems per thread, but every row a
// thread needs is streamed D rows ahead into its own 16-byte slots of a
// shared-memory ring by cp.async, so the prefetch depth costs no registers.
template <int SPB, int D, bool CYC>
__global__ void __launch_bounds__(SPB, 2)
    k_twisted_async(const float4* __restrict__ gtab, const double* __restrict__ twist,
                    double* __restrict__ X, int M, int m, int batch) {
  constexpr int SPT = 2;
  constexpr int TPD = SPB / SPT;            // threads per direction
  constexpr int NT = 2 * TPD;               // threads per CTA
  constexpr int KT = CYC ? kTwK : 3;        // float4 per table row kept in shared memory
  constexpr int NX = CYC ? 8 : 4;
  extern __shared__ __align__(128) float4 sm_tw[];
  float4* stab = sm_tw;                                          // [M][KT]
  uint4* ring = reinterpret_cast<uint4*>(stab + (size_t)M * KT);  // [D][NT]
  __shared__ double sx[TPD][SPT][NX];
  __shared__ double sT[kTwistCount];
  for (int t = threadIdx.x; t < M * KT; t += NT) cp_async16(&stab[t], &gtab[(size_t)(t / KT) * kTwK + t % KT]);
  cp_async_wait_all();
  if (threadIdx.x < kTwistCount) sT[threadIdx.x] = twist[threadIdx.x];
  __syncthreads();

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool top = warp < TPD / 32;
  const int grp = top ? warp : warp - TPD / 32;
  const int tl = grp * 32 + lane;
  const float4* tab = stab + (top ? 0 : m * KT);
  const int rows = top ? m : M - m;
  const long long ld = batch;
  const long long stepB = (top ? ld : -ld) * (long long)sizeof(double);
  const int nblk = (batch + SPB - 1) / SPB;
  const int jtop = rows - 3;
  uint4* myring = ring + tid;
  // cyclic: the border terms (q . f inward, u x_t outward) only in local rows
  // j < W, the rest of the row entries being below 2^-60
  const int W = CYC ? (int)sT[20] : 0;

  for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int s0 = blk * SPB + tl * SPT;
    const bool act = s0 < batch;
    char* p0 = reinterpret_cast<char*>(X + (top ? 0 : (long long)(M - 1) * ld) + (act ? s0 : 0));
    Lane<SPT> st;
#pragma unroll
    for (int t = 0; t < SPT; ++t) st.a1[t] = st.a2[t] = st.acc0[t] = st.acc1[t] = D2{0.f, 0.f};

    // ------------------------------------------------ inward sweep
#pragma unroll
    for (int u = 0; u < D; ++u) {
      if (u < rows) cp_async16(myring + u * NT, p0 + (long long)u * stepB);
      cp_commit();
    }
    {
      // main blocks: row j and its prefetch row j + D both exist -> no guards
      const int nmain = rows >= 2 * D ? rows / D - 1 : 0;
      char* q = p0;
      const long long pf = (long long)D * stepB;
      const float4* row = tab;
      auto block = [&](auto border) {
        constexpr bool B = decltype(border)::value;
#pragma unroll
        for (int u = 0; u < D; ++u) {
          cp_wait<D - 1>();
          double f[SPT];
          unpack2(myring[u * NT], f);
          D2 g[SPT];
          inward_row<SPT, B>(row, f, st, g);
          if (act) st_g<SPT>(q, g);
          cp_async16(myring + u * NT, q + pf);
          cp_commit();
          q += stepB;
          row += KT;
        }
      };
      if constexpr (CYC) {
        const int nb = min(nmain, (W + D - 1) / D);   // blocks that hold border rows
        int b = 0;
        for (; b < nb; ++b) block(std::true_type{});
        for (; b < nmain; ++b) block(std::false_type{});
      } else {
        for (int b = 0; b < nmain; ++b) {
#pragma unroll
          for (int u = 0; u < D; ++u) {
            cp_wait<D - 1>();
            double f[SPT];
            unpack2(myring[u * NT], f);
            D2 g[SPT];
            inward_row<SPT, false>(row, f, st, g);
            if (act) st_g<SPT>(q, g);
            cp_async16(myring + u * NT, q + pf);
            cp_commit();
            q += stepB;
            row += KT;
          }
        }
      }
      for (int j0 = nmain * D; j0 < rows; j0 += D) {
#pragma unroll
        for (int u = 0; u < D; ++u) {
          const int j = j0 + u;
          if (j < rows) {
            cp_wait<D - 1>();
            double f[SPT];
            unpack2(myring[u * NT], f);
            D2 g[SPT];
            if (CYC && j < W) inward_row<SPT, CYC>(tab + j * KT, f, st, g);
            else inward_row<SPT, false>(tab + j * KT, f, st, g);
            char* qq = p0 + (long long)j * stepB;
            if (act) st_g<SPT>(qq, g);
            if (j + D < rows) cp_async16(myring + u * NT, qq + pf);
          }
          cp_commit();
        }
      }
    }
    __threadfence();   // this thread's g stores are performed before it streams them back

    // ------------------------------------------------ meeting point (fp64)
#pragma unroll
    for (int t = 0; t < SPT; ++t) {
      if (top) {
        sx[tl][t][0] = df::to_double(st.a2[t]);
        sx[tl][t][1] = df::to_double(st.a1[t]);
        if (CYC) { sx[tl][t][4] = df::to_double(st.acc0[t]); sx[tl][t][5] = df::to_double(st.acc1[t]); }
      } else {
        sx[tl][t][2] = df::to_double(st.a1[t]);
        sx[tl][t][3] = df::to_double(st.a2[t]);
        if (CYC) { sx[tl][t][6] = df::to_double(st.acc0[t]); sx[tl][t][7] = df::to_double(st.acc1[t]); }
      }
    }
    named_barrier(1 + grp, 64);
    const double* Ti = sT + (top ? 0 : 8);
    double v0[SPT], v1[SPT], xt0[SPT], xt1[SPT];
    D2 nx0[SPT], nx1[SPT];
#pragma unroll
    for (int t = 0; t < SPT; ++t) {
      const double w0 = sx[tl][t][0], w1 = sx[tl][t][1], w2 = sx[tl][t][2], w3 = sx[tl][t][3];
      v0[t] = Ti[0] * w0 + Ti[1] * w1 + Ti[2] * w2 + Ti[3] * w3;
      v1[t] = Ti[4] * w0 + Ti[5] * w1 + Ti[6] * w2 + Ti[7] * w3;
      nx0[t] = nx1[t] = D2{0.f, 0.f};
    }
    if (CYC) {
      double ft0[SPT], ft1[SPT];
      const char* pt = reinterpret_cast<const char*>(X + (long long)M * ld + (act ? s0 : 0));
      ld_f<SPT>(pt, ft0);
      ld_f<SPT>(pt + ld * (long long)sizeof(double), ft1);
#pragma unroll
      for (int t = 0; t < SPT; ++t) {
        const double r0 = ft0[t] - (sx[tl][t][4] + sx[tl][t][6]);
        const double r1 = ft1[t] - (sx[tl][t][5] + sx[tl][t][7]);
        xt0[t] = sT[16] * r0 + sT[17] * r1;
        xt1[t] = sT[18] * r0 + sT[19] * r1;
        nx0[t] = df::from_double(-xt0[t]);
        nx1[t] = df::from_double(-xt1[t]);
      }
    }
    named_barrier(1 + grp, 64);   // partner has read sx (and f_t) before reuse / overwrite
    if (CYC && act && !top) {
      char* pt = reinterpret_cast<char*>(X + (long long)M * ld + s0);
      st_x<SPT>(pt, xt0);
      st_x<SPT>(pt + ld * (long long)sizeof(double), xt1);
    }
    {
      const int jA = top ? rows - 2 : rows - 1;
      const int jB = top ? rows - 1 : rows - 2;
      double xa[SPT], xb[SPT];
#pragma unroll
      for (int t = 0; t < SPT; ++t) {
        const D2 a = df::from_double(v0[t]), b = df::from_double(v1[t]);
        st.a1[t] = top ? a : b;
        st.a2[t] = top ? b : a;
        if (CYC) {
          const float4 cA3 = tab[jA * KT + 3], cA4 = tab[jA * KT + 4];
          const float4 cB3 = tab[jB * KT + 3], cB4 = tab[jB * KT + 4];
          xa[t] = df::to_double(df::axpy(df::axpy(a, D2{cA3.z, cA3.w}, nx0[t]), D2{cA4.x, cA4.y}, nx1[t]));
          xb[t] = df::to_double(df::axpy(df::axpy(b, D2{cB3.z, cB3.w}, nx0[t]), D2{cB4.x, cB4.y}, nx1[t]));
        } else {
          xa[t] = v0[t];
          xb[t] = v1[t];
        }
      }
      if (act) {
        st_x<SPT>(p0 + (long long)jA * stepB, xa);
        st_x<SPT>(p0 + (long long)jB * stepB, xb);
      }
    }

    // ------------------------------------------------ outward sweep, local rows jtop..0
#pragma unroll
    for (int u = 0; u < D; ++u) {
      if (jtop - u >= 0) cp_async16(myring + u * NT, p0 + (long long)(jtop - u) * stepB);
      cp_commit();
    }
    {
      const int nrows = jtop + 1;
      const int nmain = nrows >= 2 * D ? nrows / D - 1 : 0;
      char* q = p0 + (long long)jtop * stepB;
      const long long pf = (long long)D * stepB;
      const float4* row = tab + jtop * KT;
      auto block = [&](auto border) {
        constexpr bool B = decltype(border)::value;
#pragma unroll
        for (int u = 0; u < D; ++u) {
          cp_wait<D - 1>();
          const uint4 r = myring[u * NT];
          D2 g[SPT] = {D2{__uint_as_float(r.x), __uint_as_float(r.y)},
                       D2{__uint_as_float(r.z), __uint_as_float(r.w)}};
          double x[SPT];
          outward_row<SPT, B>(row, g, st, nx0, nx1, x);
          if (act) st_x<SPT>(q, x);
          cp_async16(myring + u * NT, q - pf);
          cp_commit();
          q -= stepB;
          row -= KT;
        }
      };
      // blocks b cover local rows jtop - b D .. jtop - b D - (D - 1); those wholly at
      // rows >= W skip the border term
      if constexpr (CYC) {
        const int lowest0 = jtop - (D - 1) - W;   // >= 0: block 0 is border-free
        int nfree = lowest0 < 0 ? 0 : lowest0 / D + 1;
        nfree = nfree > nmain ? nmain : nfree;
        int b = 0;
        for (; b < nfree; ++b) block(std::false_type{});
        for (; b < nmain; ++b) block(std::true_type{});
      } else {
        for (int b = 0; b < nmain; ++b) {
#pragma unroll
          for (int u = 0; u < D; ++u) {
            cp_wait<D - 1>();
            const uint4 r = myring[u * NT];
            D2 g[SPT] = {D2{__uint_as_float(r.x), __uint_as_float(r.y)},
                         D2{__uint_as_float(r.z), __uint_as_float(r.w)}};
            double x[SPT];
            outward_row<SPT, false>(row, g, st, nx0, nx1, x);
            if (act) st_x<SPT>(q, x);
            cp_async16(myring + u * NT, q - pf);
            cp_commit();
            q -= stepB;
            row -= KT;
          }
        }
      }
      for (int j0 = jtop - nmain * D; j0 >= 0; j0 -= D) {
#pragma unroll
        for (int u = 0; u < D; ++u) {
          const int j = j0 - u;
          if (j >= 0) {
            cp_wait<D - 1>();
            const uint4 r = myring[u * NT];
            D2 g[SPT] = {D2{__uint_as_float(r.x), __uint_as_float(r.y)},
                         D2{__uint_as_float(r.z), __uint_as_float(r.w)}};
            double x[SPT];
            if (CYC && j < W) outward_row<SPT, CYC>(tab + j * KT, g, st, nx0, nx1, x);
            else outward_row<SPT, false>(tab + j * KT, g, st, nx0, nx1, x);
            char* qq = p0 + (long long)j * stepB;
            if (act) st_x<SPT>(qq, x);
            if (j - D >= 0) cp_async16(myring + u * NT, qq - pf);
          }
          cp_commit();
        }
      }
    }
    cp_wait<0>();
  }
}

template <int SPB, int D, bool CYC>
cudaError_t launch_async(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  constexpr int KT = CYC ? kTwK : 3;
  const size_t smem = (size_t)p.M * KT * sizeof(float4) + (size_t)D * SPB * sizeof(uint4);
  auto kern = k_twisted_async<SPB, D, CYC>;
  const cudaError_t e = kernel_prepare((const void*)kern, smem, SPB, nullptr);
  if (e != cudaSuccess) return e;
  const int nblk = (batch + SPB - 1) / SPB;
  int grid = p.df_ctas > 0 ? p.df_ctas : 2 * p.num_sms;
  if (grid > nblk) grid = nblk;
  kern<<<grid, SPB, smem, st>>>(p.twtab, p.twist, X, p.M, p.m, batch);
  note_launch();
  return cudaGetLastError();
}

template <int SPT, int SPB, int KU, bool CYC>
cudaError_t launch(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const size_t smem = (size_t)p.M * kTwK * sizeof(float4);
  auto kern = k_twisted_df<SPT, SPB, KU, CYC>;
  const cudaError_t e = kernel_prepare((const void*)kern, smem, 2 * SPB / SPT, nullptr);
  if (e != cudaSuccess) return e;
  const int nblk = (batch + SPB - 1) / SPB;
  int grid = p.df_ctas > 0 ? p.df_ctas : 2 * p.num_sms;
  if (grid > nblk) grid = nblk;
  kern<<<grid, 2 * SPB / SPT, smem, st>>>(p.twtab, p.twist, X, p.M, p.m, batch);
  note_launch();
  return cudaGetLastError();
}

template <bool CYC>
cudaError_t dispatch(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  if (batch % 2 == 0 && p.df_async > 0) {
    if (p.df_async == 12) return launch_async<256, 12, CYC>(p, X, batch, st);
    if (p.df_async == 4) return launch_async<256, 4, CYC>(p, X, batch, st);
    if (p.df_async == 6) return launch_async<256, 6, CYC>(p, X, batch, st);
    return launch_async<256, 8, CYC>(p, X, batch, st);
  }
  if (batch % 2 == 0 && p.df_spt != 1) {
    switch (p.df_spb) {
      case 128: return p.df_ku == 4 ? launch<2, 128, 4, CYC>(p, X, batch, st)
                                    : launch<2, 128, 8, CYC>(p, X, batch, st);
      case 320: return p.df_ku == 4 ? launch<2, 320, 4, CYC>(p, X, batch, st)
                                    : launch<2, 320, 8, CYC>(p, X, batch, st);
      default:  return p.df_ku == 4 ? launch<2, 256, 4, CYC>(p, X, batch, st)
                                    : launch<2, 256, 8, CYC>(p, X, batch, st);
    }
  }
  switch (p.df_spb) {
    case 64: return launch<1, 64, 8, CYC>(p, X, batch, st);
    case 160: return launch<1, 160, 8, CYC>(p, X, batch, st);
    default: return launch<1, 128, 8, CYC>(p, X, batch, st);
  }
}

}  // namespace

cudaError_t shared_twisted_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  return p.cyclic ? dispatch<true>(p, X, batch, st) : dispatch<false>(p, X, batch, st);
}

}  // namespace pent

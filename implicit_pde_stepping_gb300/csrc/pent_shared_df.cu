// Shared-matrix batched solve in double-float arithmetic, two threads per system.
//
// Same mathematics as k_shared_thread (forward substitution L g = f and back
// substitution R x = g of "cuPentBatch – A batched pentadiagonal solver for
// NVIDIA GPUs", interleaved layout, factor once), re-planned for GB300:
//
//  * Arithmetic.  GB300 issues fp64 FMA at ~1.6/clock/SM but fp32 FMA at
//    ~115/clock/SM, so every recurrence step is done in double-float (df64.cuh)
//    on the FP32 pipe; only the final hi+lo join uses one fp64 add per point.
//  * Two threads per system (twisted factorisation, pent_factor_twisted.cu).
//    Warp w < NW sweeps rows 0..m-1 of 32 systems downwards ("top"), warp
//    w + NW sweeps rows M-1..m of the same systems upwards ("bottom").  They
//    meet in a 4x4 system (solved in fp64 from a shared-memory exchange) and
//    back-substitute outwards.  Each thread's intermediate g lives in place,
//    over f, for half as long as in a one-sided sweep, so the L2 (135 MB)
//    keeps most of it between the two sweeps and HBM sees close to the
//    two-array minimum (read f, write x).
//  * Persistent CTAs: the grid is sized to the number of SMs so that the set
//    of systems in flight, and with it the L2 working set, stays bounded.
//  * Memory: a warp touches 32 consecutive systems of one row (256 B); loads
//    are issued kU rows ahead in a register ring.  g is stored as a float pair
//    in the 8-byte slot of f and read back by the outward sweep.
//
// Cyclic plans (CYC) carry Navon's bordering (eqs. (8)–(12)) in the same pass:
// the inward sweeps accumulate q_k . f (q_k = E^{-T} h_k), the meeting point
// forms x_t = S^{-1}(f_t - q . f), and the outward sweeps subtract u_k x_t.
#include "df64.cuh"
#include "pent_internal.cuh"

namespace pent {
namespace {

using df::D2;

constexpr int kU = 8;   // rows per prefetch block (two blocks in flight)

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int SPB, bool CYC>
__global__ void __launch_bounds__(2 * SPB)
    k_shared_df(const float4* __restrict__ gtab, const double* __restrict__ twist,
                double* __restrict__ X, int M, int m, int batch) {
  extern __shared__ float4 stab[];
  __shared__ double sx[SPB][CYC ? 8 : 4];
  constexpr int NW = SPB / 32;
  const int Mb = M - m;
  {
    const int n = M * kTwK;
    for (int t = threadIdx.x; t < n; t += blockDim.x) stab[t] = gtab[t];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool top = warp < NW;
  const int grp = top ? warp : warp - NW;
  const int sl = grp * 32 + lane;
  const float4* tab = stab + (top ? 0 : (size_t)m * kTwK);
  const int rows = top ? m : Mb;
  const long long ld = batch;
  const long long step = top ? ld : -ld;
  double Ti[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) Ti[k] = twist[(top ? 0 : 8) + k];
  const int nblk = (batch + SPB - 1) / SPB;

  for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int s = blk * SPB + sl;
    const bool act = s < batch;
    double* base = X + (top ? 0 : (long long)(M - 1) * ld) + (act ? s : 0);

    // ---------------- inward sweep: g_j = r f + P g_{j-2} + Q g_{j-1}
    D2 g1{0.f, 0.f}, g2{0.f, 0.f};
    D2 acc0{0.f, 0.f}, acc1{0.f, 0.f};
    double fa[kU], fb[kU];
    auto load_f = [&](double* buf, int j0) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u;
        buf[u] = (act && j < rows) ? base[j * step] : 0.0;
      }
    };
    auto inward = [&](const double* buf, int j0) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u;
        if (j < rows) {
          const float4 c0 = tab[j * kTwK], c1 = tab[j * kTwK + 1];
          const D2 f = df::from_double(buf[u]);
          const D2 g = df::sum3p(D2{c0.x, c0.y}, f, D2{c0.z, c0.w}, g2, D2{c1.x, c1.y}, g1);
          if (CYC) {
            const float4 c2 = tab[j * kTwK + 2], c3 = tab[j * kTwK + 3];
            acc0 = df::axpy(acc0, D2{c2.z, c2.w}, f);
            acc1 = df::axpy(acc1, D2{c3.x, c3.y}, f);
          }
          if (act) *reinterpret_cast<float2*>(base + j * step) = make_float2(g.h, g.l);
          g2 = g1;
          g1 = g;
        }
      }
    };
    load_f(fa, 0);
    load_f(fb, kU);
    for (int j0 = 0; j0 < rows; j0 += 2 * kU) {
      inward(fa, j0);
      load_f(fa, j0 + 2 * kU);
      inward(fb, j0 + kU);
      load_f(fb, j0 + 3 * kU);
    }

    // ---------------- meeting point: 4x4 twist (and 2x2 border) in fp64
    // top holds g_{m-2} (g2), g_{m-1} (g1); bottom holds g~_{Mb-2} (g2) = row m+1,
    // g~_{Mb-1} (g1) = row m.  Unknowns v = (x_{m-2}, x_{m-1}, x_m, x_{m+1}).
    if (top) {
      sx[sl][0] = df::to_double(g2);
      sx[sl][1] = df::to_double(g1);
      if (CYC) { sx[sl][4] = df::to_double(acc0); sx[sl][5] = df::to_double(acc1); }
    } else {
      sx[sl][2] = df::to_double(g1);
      sx[sl][3] = df::to_double(g2);
      if (CYC) { sx[sl][6] = df::to_double(acc0); sx[sl][7] = df::to_double(acc1); }
    }
    named_barrier(1 + grp, 64);
    const double w0 = sx[sl][0], w1 = sx[sl][1], w2 = sx[sl][2], w3 = sx[sl][3];
    // my two unknowns: top -> (x_{m-2}, x_{m-1}), bottom -> (x_m, x_{m+1})
    const double v0 = Ti[0] * w0 + Ti[1] * w1 + Ti[2] * w2 + Ti[3] * w3;
    const double v1 = Ti[4] * w0 + Ti[5] * w1 + Ti[6] * w2 + Ti[7] * w3;
    D2 nxt0{0.f, 0.f}, nxt1{0.f, 0.f};   // -x_t0, -x_t1 as double-floats (cyclic)
    if (CYC) {
      const double a0 = sx[sl][4] + sx[sl][6], a1 = sx[sl][5] + sx[sl][7];
      const double ft0 = act ? X[(long long)M * ld + s] : 0.0;
      const double ft1 = act ? X[(long long)(M + 1) * ld + s] : 0.0;
      const double t0 = ft0 - a0, t1 = ft1 - a1;
      const double xt0 = twist[16] * t0 + twist[17] * t1;
      const double xt1 = twist[18] * t0 + twist[19] * t1;
      nxt0 = df::from_double(-xt0);
      nxt1 = df::from_double(-xt1);
      named_barrier(1 + grp, 64);       // both threads have read f_t before it is replaced
      if (act && !top) {
        X[(long long)M * ld + s] = xt0;
        X[(long long)(M + 1) * ld + s] = xt1;
      }
    } else {
      named_barrier(1 + grp, 64);       // sx may be reused by the next block
    }
    // local rows rows-2 (value v0 for top: x_{m-2}; bottom: x_{m+1} is v1) ...
    // top: local m-2 <- v0, m-1 <- v1.   bottom: local Mb-1 (row m) <- v0, Mb-2 (row m+1) <- v1.
    D2 y1, y2;   // y_{j+1}, y_{j+2} in local order
    {
      const D2 a = df::from_double(v0), b = df::from_double(v1);
      if (top) { y1 = a; y2 = b; }     // j = m-3: y_{m-2} = v0, y_{m-1} = v1
      else     { y1 = b; y2 = a; }     // j = Mb-3: y~_{Mb-2} = x_{m+1} = v1, y~_{Mb-1} = x_m = v0
      const int jA = top ? rows - 2 : rows - 1;   // local row holding v0
      const int jB = top ? rows - 1 : rows - 2;   // local row holding v1
      D2 xa = a, xb = b;
      if (CYC) {
        const float4 cA3 = tab[jA * kTwK + 3], cA4 = tab[jA * kTwK + 4];
        const float4 cB3 = tab[jB * kTwK + 3], cB4 = tab[jB * kTwK + 4];
        xa = df::axpy(df::axpy(xa, D2{cA3.z, cA3.w}, nxt0), D2{cA4.x, cA4.y}, nxt1);
        xb = df::axpy(df::axpy(xb, D2{cB3.z, cB3.w}, nxt0), D2{cB4.x, cB4.y}, nxt1);
      }
      if (act) {
        base[jA * step] = df::to_double(xa);
        base[jB * step] = df::to_double(xb);
      }
    }

    // ---------------- outward sweep: y_j = g_j + C y_{j+1} + D y_{j+2}
    float2 ga[kU], gb[kU];
    auto load_g = [&](float2* buf, int j0) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 - u;
        buf[u] = (act && j >= 0) ? *reinterpret_cast<const float2*>(base + j * step)
                                 : make_float2(0.f, 0.f);
      }
    };
    auto outward = [&](const float2* buf, int j0) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 - u;
        if (j >= 0) {
          const float4 c1 = tab[j * kTwK + 1], c2 = tab[j * kTwK + 2];
          const D2 y = df::sum3(D2{buf[u].x, buf[u].y}, D2{c1.z, c1.w}, y1, D2{c2.x, c2.y}, y2);
          D2 x = y;
          if (CYC) {
            const float4 c3 = tab[j * kTwK + 3], c4 = tab[j * kTwK + 4];
            x = df::axpy(df::axpy(x, D2{c3.z, c3.w}, nxt0), D2{c4.x, c4.y}, nxt1);
          }
          if (act) __stcs(base + j * step, df::to_double(x));
          y2 = y1;
          y1 = y;
        }
      }
    };
    const int jstart = rows - 3;
    load_g(ga, jstart);
    load_g(gb, jstart - kU);
    for (int j0 = jstart; j0 >= 0; j0 -= 2 * kU) {
      outward(ga, j0);
      load_g(ga, j0 - 2 * kU);
      outward(gb, j0 - kU);
      load_g(gb, j0 - 3 * kU);
    }
  }
}

template <int SPB, bool CYC>
cudaError_t launch(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const size_t smem = (size_t)p.M * kTwK * sizeof(float4);
  auto kern = k_shared_df<SPB, CYC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nblk = (batch + SPB - 1) / SPB;
  int grid = p.df_ctas > 0 ? p.df_ctas : p.num_sms;
  if (grid > nblk) grid = nblk;
  kern<<<grid, 2 * SPB, smem, st>>>(p.twtab, p.twist, X, p.M, p.m, batch);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

size_t shared_df_smem_bytes(int M) { return (size_t)M * kTwK * sizeof(float4); }

cudaError_t shared_thread_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const int spb = p.df_spb;
  if (p.cyclic) {
    if (spb == 64) return launch<64, true>(p, X, batch, st);
    if (spb == 96) return launch<96, true>(p, X, batch, st);
    return launch<128, true>(p, X, batch, st);
  }
  if (spb == 64) return launch<64, false>(p, X, batch, st);
  if (spb == 96) return launch<96, false>(p, X, batch, st);
  if (spb == 160) return launch<160, false>(p, X, batch, st);
  return launch<128, false>(p, X, batch, st);
}

}  // namespace pent

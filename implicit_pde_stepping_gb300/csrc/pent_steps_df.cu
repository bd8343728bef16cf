// Persistent multi-step kernel: nsteps of a periodic time scheme in one launch,
// the state of every system held in registers from the first step to the last.
//
// Each step is the partitioned double-float cyclic solve of pent_split_df.cu
// (forward and back substitution of "cuPentBatch – A batched pentadiagonal
// solver for NVIDIA GPUs" per chunk of L rows, chunk boundary states by the
// truncated parallel scan, Navon's bordering, eqs. (8)–(12), for the two
// periodic rows), but the right-hand side of step n+1 is taken from the
// registers that hold the result of step n, so a system touches memory twice
// in the whole launch: one load of C^0, one store of C^nsteps.  Schemes:
//   hyperdiffusion (eq. (4)):      A C^{n+1} = C^n;
//   Cahn–Hilliard (eq. (2)):       A C^{n+1} = C^n + k2 D2[(C^n)^3 - C^n];
//   Crank–Nicolson (eqs. (5)–(6)): A C^{n+1} = (2I - A) C^n, i.e.
//                                  C^{n+1} = 2 A^{-1} C^n - C^n.
// Between steps the state stays a double-float (hi, lo) pair, renormalised
// after every step; it is rounded to fp64 once, at the final store.  In the
// 8-row groups where a chunk's responses to a neighbour's state are below 2^-24
// in every chunk (found when the plan is built: the last rows of a chunk for the
// incoming state, the first rows for the outgoing one, when the couplings decay
// fast), those correction terms take one FMA into the low word.
//
// Cross-chunk data per step: the Cahn–Hilliard right-hand side of a chunk's
// first and last rows needs C of the neighbouring rows, exchanged through
// shared memory (first and last value of every chunk); the two periodic rows
// M = N-2 and M+1 = N-1 are kept by the system's chunk-0 thread in shared
// memory.  Crank–Nicolson keeps C^n of every row in shared memory for the
// final 2y - C.
//
// Launched only when the plan's chunk couplings are truncated (T > 0); the
// exact serial chunk scan stays with the one-step kernel.
//
// Range: as in the one-step kernel, each system is scaled by the power of two
// that puts the largest entry of C^0 in [1, 2) (the Cahn–Hilliard cubic then
// carries 2^(2s)).  The scale is kept for all steps; the kernel watches the
// state, and a system that grows beyond 2^8 in these units (only the explicit
// Cahn–Hilliard cubic can make it grow, when |C| is well above 1) is not
// stored: like the systems outside the scaled path's window, it is stepped
// natively in fp64 by one thread from its untouched C^0.
#include <type_traits>

#include "cp_async.cuh"
#include "df64.cuh"
#include "fg.cuh"
#include "pent_internal.cuh"
#include "pent_native.cuh"

namespace pent {
namespace {

using df::D2;

constexpr int kStepHyper = 0;
constexpr int kStepCH = 1;
constexpr int kStepCN = 2;

// u = q c^3 - c for the scaled state c = C 2^-s, q = 2^(2s)
__device__ __forceinline__ D2 cubic_minus(D2 c, float q) {
  const D2 c3 = df::mul(df::mul(c, c), c);
  return df::add(D2{c3.h * q, c3.l * q}, df::neg(c));
}

// C_i + k2 (u_{i-1} - 2 u_i + u_{i+1})
__device__ __forceinline__ D2 ch_rhs(D2 c, D2 um, D2 u0, D2 up, D2 k2) {
  const D2 lap = df::add(df::add(um, up), D2{-2.f * u0.h, -2.f * u0.l});
  return df::add(c, df::mul(k2, lap));
}

// a + b = s + e for |a| >= |b| (Dekker's Fast2Sum, three operations)
__device__ __forceinline__ void quick_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

__device__ __forceinline__ D2 pick(bool p, D2 a, D2 b) { return D2{p ? a.h : b.h, p ? a.l : b.l}; }
__device__ __forceinline__ float2 pack(D2 a) { return make_float2(a.h, a.l); }
__device__ __forceinline__ D2 unpack(float2 a) { return D2{a.x, a.y}; }

// y += A x for a row-major 2x2 A of double-float pairs
__device__ __forceinline__ void mv2d(const float2* A, D2 x0, D2 x1, D2& y0, D2& y1) {
  y0 = df::sum3(y0, unpack(A[0]), x0, unpack(A[1]), x1);
  y1 = df::sum3(y1, unpack(A[2]), x0, unpack(A[3]), x1);
}

// Chunks dup_lo < c <= dup_hi have row and chunk tables bitwise equal to chunk
// dup_lo's (found when the plan was built) and share its row-table slot.
__host__ __device__ __forceinline__ int table_slot(int c, int lo, int hi) {
  return c <= lo ? c : (c <= hi ? lo : c - (hi - lo));
}

// Shared memory of one CTA (bytes), in the order the kernel carves it; the row
// tables in nslot slots (nslot = P without shared slots).
__host__ __device__ inline size_t steps_smem(int L, int P, int SB, int rhs, int nslot) {
  size_t b = (size_t)nslot * (L * kSpK + 1) * sizeof(float4);    // row tables
  b += ((size_t)P * kSpChunk + 2 * (size_t)SB * P * 2 + (size_t)SB * 8) * sizeof(double);
  b += kSpExtra * sizeof(float2);                                   // extras as (hi, lo)
  if (rhs == kStepCH) b += ((size_t)SB * P * 2 + SB) * sizeof(float2);   // halo, C_{M-1}
  if (rhs == kStepCN) b += (size_t)L * SB * P * sizeof(float2);          // C^n of every row
  b += 2 * (size_t)SB * sizeof(uint32_t);                                // largest |C^0| bits, growth flags
  return b;
}

template <int L, int SB, int MAXT, int RHS, bool CHEAP>
__global__ void __launch_bounds__(MAXT, 1)
    k_steps_df(const float4* __restrict__ growtab, const float2* __restrict__ gchunk,
               const double* __restrict__ gextra, double* __restrict__ X, int M, int P, int batch,
               int nsteps, double k2d, int2 cheap, const NativeTabs nt, int dup_lo, int dup_hi) {
  constexpr bool CH = RHS == kStepCH;
  constexpr bool CN = RHS == kStepCN;
  constexpr int K4 = kSpK;
  constexpr int CS = L * K4 + 1;              // chunk stride (float4), padded
  constexpr int SG = SB / 8;                  // system groups of 8 per CTA
  constexpr int LG = 8;                       // rows per load group
  extern __shared__ float4 smem4[];
  float4* rtab = smem4;                                              // [P][CS]
  const int nslot = P - (dup_hi - dup_lo);
  float2* ctab = reinterpret_cast<float2*>(rtab + (size_t)nslot * CS);   // [P][kSpChunk] (hi, lo)
  float2* sE = ctab + (size_t)P * kSpChunk;      // [SB][P][2] local forward end values
  float2* sW = sE + (size_t)SB * P * 2;          // [SB][P][2] w_c
  float2* sX = sW + (size_t)SB * P * 2;         // [SB][8] y at 4 rows, x_t, tail state (hi, lo)
  float2* sXe = sX + (size_t)SB * 8;             // [kSpExtra] the plan's extras as (hi, lo)
  float2* sH = sXe + kSpExtra;                   // CH: [SB][P][2] first, last C
  float2* sA = sH + (CH ? (size_t)SB * P * 2 : 0);               // CH: [SB] C_{M-1}
  float2* sC = sA + (CH ? (size_t)SB : 0);                       // CN: [L][SB * P] C^n
  uint32_t* smax = reinterpret_cast<uint32_t*>(sC + (CN ? (size_t)L * SB * P : 0));   // [SB]
  uint32_t* sgrow = smax + SB;                                                          // [SB]

  for (int t = threadIdx.x; t < P * L * K4; t += blockDim.x) {
    const int row = t / K4, k = t % K4, cc = row / L;
    if (cc > dup_lo && cc <= dup_hi) continue;                     // shares chunk dup_lo's slot
    cp_async16(&rtab[table_slot(cc, dup_lo, dup_hi) * CS + (row % L) * K4 + k], &growtab[(size_t)row * kSpK + k]);
  }
  for (int t = threadIdx.x; t < P * kSpChunk / 2; t += blockDim.x) cp_async16(&ctab[2 * t], &gchunk[2 * t]);
  if (threadIdx.x < kSpExtra) sXe[threadIdx.x] = pack(df::from_double(gextra[threadIdx.x]));
  for (int t = threadIdx.x; t < SB; t += blockDim.x) smax[t] = sgrow[t] = 0u;
  cp_async_wait_all();
  __syncthreads();
  const int T = (int)gextra[18];

  const int tid = threadIdx.x, nthr = SB * P;
  const int lane = tid & 31, w = tid >> 5;
  const int sys = (w % SG) * 8 + (lane & 7);
  const int c = (w / SG) * 4 + (lane >> 3);
  const int row0 = c * L;
  const float4* ctb = rtab + (size_t)table_slot(c, dup_lo, dup_hi) * CS;
  const float2* ct = ctab + (size_t)c * kSpChunk;
  const long long ld = batch;
  const int nblk = (batch + SB - 1) / SB;
  const bool ownM2 = row0 <= M - 2 && M - 2 < row0 + L;
  const bool ownM1 = row0 <= M - 1 && M - 1 < row0 + L;
  // x_t correction only in the chunks where it is not negligible
  const int reach = (int)gextra[19];
  const bool needU = c < reach || c > (M - 1) / L - reach;
  float2* xc = sX + (size_t)sys * 8;
  auto ex = [&](int k) { return unpack(sXe[k]); };

  for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int s = blk * SB + sys;
    const bool act = s < batch;
    double* p = X + (long long)row0 * ld + (act ? s : 0);

    // ---- the system's scale: its largest |C^0| (one pass over the rows; the
    // loads below find them in cache)
    {
      // magnitude word: largest high word, bit 0 set if any low word is nonzero
      uint32_t mx = 0u, nz = 0u;
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (act && row0 + j < M) {
          const double v = p[j * ld];
          mx = max(mx, fg::mag_bits(v));
          nz |= (uint32_t)__double2loint(v);
        }
      if (c == 0 && act) {
        const double v0 = X[(long long)M * ld + s], v1 = X[(long long)(M + 1) * ld + s];
        mx = max(mx, fg::mag_pair(v0, v1, nz));
      }
      atomicMax(&smax[sys], mx | (nz != 0u ? 1u : 0u));
    }
    __syncthreads();
    const uint32_t emax = smax[sys] >> 20;
    const bool fast = emax >= fg::kEMin && emax <= (CH ? fg::kEMaxCH : fg::kEMax);
    // an all-zero state stays zero under every step: nothing to store
    const bool keep = smax[sys] == 0u;
    const bool native = act && !fast && !keep;
    const uint32_t esys = fast ? emax : 1023u;
    const uint32_t ioff = fg::in_offset(esys), ooff = fg::out_offset(esys);
    const float q = fg::cubic_scale(esys);
    auto sdf = [&](double x) {
      float h, lo;
      fg::split(x, ioff, h, lo);
      return D2{h, lo};
    };

    // ---- C^0: rows of this chunk into registers (padding rows 0), tail into shared memory
    D2 v[L];
#pragma unroll
    for (int j0 = 0; j0 < L; j0 += LG) {
      double fv[LG];
#pragma unroll
      for (int u = 0; u < LG; ++u) fv[u] = (act && row0 + j0 + u < M) ? p[(j0 + u) * ld] : 0.0;
#pragma unroll
      for (int u = 0; u < LG; ++u) v[j0 + u] = sdf(fv[u]);
    }
    if (c == 0) {
      xc[6] = pack(sdf(act ? X[(long long)M * ld + s] : 0.0));
      xc[7] = pack(sdf(act ? X[(long long)(M + 1) * ld + s] : 0.0));
    }
    __syncthreads();
    if (c == 0) smax[sys] = sgrow[sys] = 0u;                // next block (ordered by the next barrier)
    float grow = 0.f;                                       // largest |state| after any step

    for (int n = 0; n < nsteps; ++n) {
      const D2 ct0 = unpack(xc[6]), ct1 = unpack(xc[7]);   // C at rows M, M+1
      D2 ft0 = ct0, ft1 = ct1;                             // right-hand side of the two periodic rows

      // ---- 1. forward substitution with this step's right-hand side (zero incoming state)
      {
        D2 a1{0.f, 0.f}, a2{0.f, 0.f};
        if constexpr (CH) {
          float2* hs = sH + ((size_t)sys * P + c) * 2;
          hs[0] = pack(v[0]);
          hs[1] = pack(v[L - 1]);
          if (ownM1) {
            D2 cm1 = v[0];
#pragma unroll
            for (int j = 0; j < L; ++j) cm1 = pick(row0 + j == M - 1, v[j], cm1);
            sA[sys] = pack(cm1);
          }
          __syncthreads();                                  // halos published
          const D2 k2 = df::from_double(k2d);
          if (c == 0) {                                     // rows M, M+1 need C_{M-1}, C_0
            const D2 cA = unpack(sA[sys]);
            const D2 uA = cubic_minus(cA, q), uB = cubic_minus(ct0, q), uC = cubic_minus(ct1, q);
            const D2 uD = cubic_minus(v[0], q);
            ft0 = ch_rhs(ct0, uA, uB, uC, k2);
            ft1 = ch_rhs(ct1, uB, uC, uD, k2);
          }
          const D2 lh = c == 0 ? ct1 : unpack(sH[((size_t)sys * P + c - 1) * 2 + 1]);
          D2 rh = c + 1 < P ? unpack(sH[((size_t)sys * P + c + 1) * 2]) : D2{0.f, 0.f};
          rh = pick(row0 + L == M, ct0, rh);
          D2 cc = v[0];
          D2 um = cubic_minus(lh, q), u0 = cubic_minus(cc, q);
#pragma unroll
          for (int j = 0; j < L; ++j) {
            D2 cn = (j + 1 < L) ? v[j + 1 < L ? j + 1 : j] : rh;
            cn = pick(row0 + j + 1 == M, ct0, cn);          // row M is periodic state
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
#pragma unroll
          for (int j = 0; j < L; ++j) {
            const D2 f = v[j];                              // padding rows hold 0
            if constexpr (CN) sC[(size_t)j * nthr + tid] = pack(f);
            const float4 c0 = ctb[j * K4];
            const float4 c1 = ctb[j * K4 + 1];
            const D2 g = df::sum3p(D2{c0.x, c0.y}, f, D2{c0.z, c0.w}, a2, D2{c1.x, c1.y}, a1);
            v[j] = g;
            a2 = a1;
            a1 = g;
          }
        }
      }
      float2* eo = sE + ((size_t)sys * P + c) * 2;
      eo[0] = pack(v[L - 2]);
      eo[1] = pack(v[L - 1]);
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
      const D2 xs0 = v[0], xs1 = v[1];
      D2 xm2{0.f, 0.f}, xm1{0.f, 0.f};
      if (ownM2 || ownM1) {
        D2 a = v[0], b = v[0];
#pragma unroll
        for (int j = 0; j < L; ++j) {
          a = pick(row0 + j == M - 2, v[j], a);
          b = pick(row0 + j == M - 1, v[j], b);
        }
        xm2 = a;
        xm1 = b;
      }

      // ---- 2. chunk boundary states s_c, t_c (truncated parallel scan), in
      // double-float on the FP32 pipe: in fp64 these few operations per thread
      // queue on the slow fp64 pipe between two barriers, with every warp waiting
      D2 s0{0.f, 0.f}, s1{0.f, 0.f}, t0{0.f, 0.f}, t1{0.f, 0.f};
      __syncthreads();                                      // e_c published
      {
        const float2* E = sE + (size_t)sys * P * 2;
        for (int k = 1; k <= T && k <= c; ++k) {
          const D2 ea = unpack(E[2 * (c - k)]), eb = unpack(E[2 * (c - k) + 1]);
          if (k == 1) { s0 = df::add(s0, ea); s1 = df::add(s1, eb); }
          else mv2d(ct + 12 + 4 * (k - 2), ea, eb, s0, s1);
        }
      }
      D2 w0 = xs0, w1 = xs1;
      mv2d(ct + 4, s0, s1, w0, w1);
      float2* wo = sW + ((size_t)sys * P + c) * 2;
      wo[0] = pack(w0);
      wo[1] = pack(w1);
      __syncthreads();                                      // w_c published
      {
        const float2* Wv = sW + (size_t)sys * P * 2;
        for (int k = 0; k < T && c + 1 + k < P; ++k) {
          const D2 wa = unpack(Wv[2 * (c + 1 + k)]), wb = unpack(Wv[2 * (c + 1 + k) + 1]);
          if (k == 0) { t0 = df::add(t0, wa); t1 = df::add(t1, wb); }
          else mv2d(ct + 24 + 4 * (k - 1), wa, wb, t0, t1);
        }
      }
      if (c == 0) {
        D2 y0 = w0, y1 = w1;
        mv2d(ct + 8, t0, t1, y0, y1);
        xc[2] = pack(y0);
        xc[3] = pack(y1);
      }
      // y at rows M-2, M-1 and the border solve below in double-float as well
      if (ownM2) xc[0] = pack(df::sum3(df::sum3(xm2, ex(10), s0, ex(11), s1), ex(14), t0, ex(15), t1));
      if (ownM1) xc[1] = pack(df::sum3(df::sum3(xm1, ex(12), s0, ex(13), s1), ex(16), t0, ex(17), t1));
      __syncthreads();                                      // y at rows M-2, M-1, 0, 1 published
      // periodic rows: x_t = S^{-1}(f_t - H^T y)   (eq. (12)); then the next tail state
      if (c == 0) {
        const D2 y0 = unpack(xc[0]), y1 = unpack(xc[1]), y2 = unpack(xc[2]), y3 = unpack(xc[3]);
        const D2 r0 = df::sum3(df::mul(ex(4), y0), ex(5), y1, ex(6), y2);
        const D2 r1 = df::sum3(df::mul(ex(7), y1), ex(8), y2, ex(9), y3);
        const D2 d0 = df::add(ft0, df::neg(r0)), d1 = df::add(ft1, df::neg(r1));
        const D2 u0 = df::sum3(D2{0.f, 0.f}, ex(0), d0, ex(1), d1);
        const D2 u1 = df::sum3(D2{0.f, 0.f}, ex(2), d0, ex(3), d1);
        xc[4] = pack(u0);
        xc[5] = pack(u1);
        xc[6] = CN ? pack(df::add(D2{2.f * u0.h, 2.f * u0.l}, df::neg(ct0))) : pack(u0);
        xc[7] = CN ? pack(df::add(D2{2.f * u1.h, 2.f * u1.l}, df::neg(ct1))) : pack(u1);
      }
      __syncthreads();                                      // x_t published
      const D2 xt0 = unpack(xc[4]), xt1 = unpack(xc[5]);

      // ---- 3. x = x' + M1 s0 + M2 s1 + K1 t0 + K2 t1 - u0 x_t0 - u1 x_t1: the next state
      {
        const D2 S0 = s0, S1 = s1, T0 = t0, T1 = t1;
        const D2 X0 = df::neg(xt0), X1 = df::neg(xt1);
        // one 8-row group; mode 1: the M responses are below 2^-24 in every chunk
        // here, mode 2: the K responses are, so those terms go to the low word alone
        // (dropped cross terms and rounding below about 3 * 2^-48 of the state)
        auto corr_group = [&](auto gi, auto mode) {
          constexpr int g = decltype(gi)::value, md = decltype(mode)::value;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = g * 8 + u;
            const float4 c3 = ctb[j * K4 + 3], c4 = ctb[j * K4 + 4];
            D2 x = v[j];
            if constexpr (md == 1) {
              x.l = __fmaf_rn(c3.x, S0.h, x.l);
              x.l = __fmaf_rn(c3.z, S1.h, x.l);
            } else {
              x = df::axpy(x, D2{c3.x, c3.y}, S0);
              x = df::axpy(x, D2{c3.z, c3.w}, S1);
            }
            if constexpr (md == 2) {
              x.l = __fmaf_rn(c4.x, T0.h, x.l);
              x.l = __fmaf_rn(c4.z, T1.h, x.l);
            } else {
              x = df::axpy(x, D2{c4.x, c4.y}, T0);
              x = df::axpy(x, D2{c4.z, c4.w}, T1);
            }
            v[j] = x;
          }
        };
        // K responses fall towards a chunk's start, M responses towards its end: the
        // first half of the groups may take mode 2, the second half mode 1
        auto corr = [&](auto gi) {
          [[maybe_unused]] constexpr int g = decltype(gi)::value;
          using full = std::integral_constant<int, 0>;
          if constexpr (!CHEAP) {
            corr_group(gi, full{});
          } else if constexpr (g < L / 16) {
            if (g < cheap.x) corr_group(gi, std::integral_constant<int, 2>{});
            else corr_group(gi, full{});
          } else {
            if (g >= cheap.y) corr_group(gi, std::integral_constant<int, 1>{});
            else corr_group(gi, full{});
          }
        };
        static_assert(L == 16 || L == 32, "chunks of 16 or 32 rows");
        corr(std::integral_constant<int, 0>{});
        corr(std::integral_constant<int, 1>{});
        if constexpr (L == 32) {
          corr(std::integral_constant<int, 2>{});
          corr(std::integral_constant<int, 3>{});
        }
        if (needU) {
#pragma unroll
          for (int j = 0; j < L; ++j) {
            const float4 c1 = ctb[j * K4 + 1], c5 = ctb[j * K4 + 5];
            const D2 x = df::axpy(v[j], D2{c1.z, c1.w}, X0);
            v[j] = df::axpy(x, D2{c5.x, c5.y}, X1);
          }
        }
#pragma unroll
        for (int j = 0; j < L; ++j) {
          D2 x = v[j];
          if constexpr (CN) x = df::add(D2{2.f * x.h, 2.f * x.l}, df::neg(unpack(sC[(size_t)j * nthr + tid])));
          if (row0 + j >= M) x = D2{0.f, 0.f};
          // renormalise (h, l) so that |l| <= ulp(h)/2: carried unnormalised from
          // step to step, the low word grows and its own rounding error with it
          // (|l| is a few ulps of h at most, so Fast2Sum is exact here)
          float sh, sl;
          quick_two_sum(x.h, x.l, sh, sl);
          v[j] = D2{sh, sl};
          grow = fmaxf(grow, fabsf(sh));
        }
      }
    }

    // ---- C^nsteps back to memory, unless the system outgrew its scale
    if (c == 0) grow = fmaxf(grow, fmaxf(fabsf(unpack(xc[6]).h), fabsf(unpack(xc[7]).h)));
    if (!(grow <= 256.f)) atomicOr(&sgrow[sys], 1u);      // also catches NaN
    __syncthreads();
    const bool nat = native || (act && !keep && sgrow[sys] != 0u);
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (act && !nat && !keep && row0 + j < M) __stcs(p + j * ld, fg::join(v[j].h, v[j].l, ooff));
    if (c == 0 && act && !nat && !keep) {
      const D2 t0 = unpack(xc[6]), t1 = unpack(xc[7]);
      X[(long long)M * ld + s] = fg::join(t0.h, t0.l, ooff);
      X[(long long)(M + 1) * ld + s] = fg::join(t1.h, t1.l, ooff);
    }
    // systems outside the scaled path: one thread steps the column natively
    if (nat && c == 0) {
      if constexpr (CH) native_ch_col(nt, X + s, M + 2, (size_t)ld, k2d, nsteps);
      else if constexpr (CN) native_cn_col(nt, X + s, M + 2, (size_t)ld, nsteps);
      else native_hyper_col(nt, X + s, M, (size_t)ld, nsteps);
    }
    __syncthreads();                                        // shared state reused by the next block
  }
}

template <int L, int SB, int RHS, bool CHEAP>
cudaError_t launch(const pent_plan_s& p, double* X, int batch, int nsteps, double k2,
                   cudaStream_t st) {
  const int P = p.sp_P;
  const int nslot = P - (p.dup_hi - p.dup_lo);
  const size_t smem = steps_smem(L, P, SB, RHS, nslot);
  auto kern = k_steps_df<L, SB, 512, RHS, CHEAP>;
  int per_sm = 0;
  const cudaError_t e = kernel_prepare((const void*)kern, smem, SB * P, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int nblk = (batch + SB - 1) / SB;
  int grid = p.df_ctas > 0 ? p.df_ctas : per_sm * p.num_sms;
  if (grid > nblk) grid = nblk;
  const NativeTabs nt{p.coef64, p.tail64, p.bands};
  kern<<<grid, SB * P, smem, st>>>(p.sptab, p.spchunk_df, p.spextra, X, p.M, P, batch, nsteps, k2,
                                   make_int2(p.cheap_k, p.cheap_m), nt, p.dup_lo, p.dup_hi);
  note_launch();
  return cudaGetLastError();
}

// 16 systems per CTA when they fit (one copy of the tables serves more
// systems) and the batch still gives every SM a CTA; else 8.
template <int RHS>
cudaError_t launch_kind(const pent_plan_s& p, double* X, int batch, int nsteps, double k2,
                        cudaStream_t st) {
  if (p.sp_L == 16) return launch<16, 8, RHS, false>(p, X, batch, nsteps, k2, st);
  // the low-word correction groups only where the plan found some (the kernel that
  // has them is slower when none apply: measured 4% for Crank–Nicolson, 6% for
  // Cahn–Hilliard)
  const bool cheap = p.cheap_k > 0 || p.cheap_m < p.sp_L / 8;
  const bool fits16 = p.sp_P <= 32 && steps_smem(32, p.sp_P, 16, RHS, p.sp_P - (p.dup_hi - p.dup_lo)) <= kStepsSmemMax;
  const bool wide = p.steps_sb == 16 ? fits16 : p.steps_sb == 8 ? false : fits16 && batch > 16 * p.num_sms;
  if (wide)
    return cheap ? launch<32, 16, RHS, true>(p, X, batch, nsteps, k2, st)
                 : launch<32, 16, RHS, false>(p, X, batch, nsteps, k2, st);
  return cheap ? launch<32, 8, RHS, true>(p, X, batch, nsteps, k2, st)
               : launch<32, 8, RHS, false>(p, X, batch, nsteps, k2, st);
}

}  // namespace

bool steps_supported(const pent_plan_s& p, int kind) {
  if (!p.cyclic || !p.split_ok || p.sp_T <= 0 || p.sp_P > kSpMaxChunks) return false;
  const int rhs = kind == 1 ? kStepCH : kind == 2 ? kStepCN : kStepHyper;
  return steps_smem(p.sp_L, p.sp_P, 8, rhs, p.sp_P - (p.dup_hi - p.dup_lo)) <= kStepsSmemMax && 8 * p.sp_P <= 512;
}

cudaError_t steps_df(const pent_plan_s& p, double* X, int batch, int nsteps, int kind, double k2,
                     cudaStream_t st) {
  if (kind == 1) return launch_kind<kStepCH>(p, X, batch, nsteps, k2, st);
  if (kind == 2) return launch_kind<kStepCN>(p, X, batch, nsteps, 0.0, st);
  return launch_kind<kStepHyper>(p, X, batch, nsteps, 0.0, st);
}

}  // namespace pent

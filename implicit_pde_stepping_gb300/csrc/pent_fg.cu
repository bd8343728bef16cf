// Partitioned shared-matrix solve in fixed-grid double-float.
//
// The mathematics are those of the partitioned double-float kernel
// (pent_split_df.cu, tables from pent_factor_split.cu): forward substitution
// L g = f and back substitution R x = g of "cuPentBatch – A batched
// pentadiagonal solver for NVIDIA GPUs" (factor once, interleaved layout),
// with every system cut into P chunks of L rows, one thread per chunk, so that
// the whole system stays in registers and memory sees f once and x once:
//   1. each chunk runs both sweeps locally with zero boundary values -> x';
//   2. the chunk boundary states s_c (g entering) and t_c (x leaving) follow
//      from the T nearest chunks' end values (the plan kept every coupling
//      above 2^-64), on the same grid;
//   3. x = x' + M1 s0 + M2 s1 + K1 t0 + K2 t1, joined to fp64 and stored.
// What differs is the arithmetic of all three steps: values live on a per-system fixed grid (fg.cuh), so a
// multiply-add takes six FP32 instructions instead of twelve.  The grid needs
// a scale, so every system is first scaled by the power of two that brings
// its largest |f| into [1, 2) (an exact operation folded into the fp64
// conversions); the plan bounds every intermediate value of the solve for
// such a right-hand side (rows sums of |L^-1 R|, |A^-1| and the chunk-local
// |R^-1|) and picks the grid from that bound.  The scale also gives the
// kernel the full fp64 exponent range: all-zero systems are left as they are
// (zero is their solution), systems
// whose largest entry is at or above 2^1001 are converted out at 2^1000 and
// scaled back in fp64, and only systems whose largest entry is below 2^-860
// or not finite are left to a native fp64 solve of the column by one thread
// (a sequential fp64 sweep: on GB300 it takes about as long as the whole
// batch's solve, so it is kept for those inputs alone).
//
// Correction terms whose responses are below 2^-24 over a whole 8-row group
// of every chunk go to the low word with one FMA, and those below 2^-56 are
// dropped (both decided when the plan is built).
//
// Warp layout: 8 consecutive systems x 4 chunks per warp, so every load or
// store instruction moves four 64-byte runs of one row each.  A CTA holds 8
// systems x P chunks; the grid is persistent, two CTAs per SM, and every block
// of 8 systems after a CTA's first comes from an atomic queue in the plan.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <type_traits>
#include <vector>

#include "cp_async.cuh"
#include "df64.cuh"
#include "fg.cuh"
#include "pent_internal.cuh"
#include "pent_native.cuh"
#include "tma.cuh"

namespace pent {
namespace {

using df::D2;

using fg::kEMin;
using fg::kEMax;

struct FgArgs {
  const float4* rowtab;     // [Mpad][kSpK] double-float row tables
  const float2* chunk_df;   // [P][kSpChunk] chunk couplings as (hi, lo) pairs
  const double* coef64;     // native tables for the fallback
  const double* tail64;
  double* X;
  int* err;                 // set to 1 if a tile copy never completed
  unsigned* sched;          // {next block, CTAs done}: the block queue, zero at launch
  int M, P, batch, T;
  int dup_lo, dup_hi;       // chunks dup_lo < c <= dup_hi read chunk dup_lo's row tables
  int RS, BR;               // staged rows (multiple of BR) and rows per TMA box
  float B;                  // grid bias 1.5 * 2^(k+23)
  int gm_full, gm_none;     // M1/M2: full terms in groups < gm_full, low word below gm_none
  int gk_none, gk_full;     // K1/K2: none in groups < gk_none, low word below gk_full
};

// Shared-memory slot of chunk c's row tables: chunks inside the run of
// bitwise-equal tables share the run's first slot.
__host__ __device__ __forceinline__ int row_slot(int c, int lo, int hi) {
  return c <= lo ? c : (c <= hi ? lo : c - (hi - lo));
}

// Bytes of the f tile: RS rows of SB systems (fp64).
__host__ __device__ __forceinline__ size_t tile_bytes(int RS, int SB) { return (size_t)RS * SB * sizeof(double); }

template <int L, int SB, int MAXT, bool TMA>
__global__ void __launch_bounds__(MAXT, (MAXT <= 256 ? 2 : 1))
    k_fg(const __grid_constant__ CUtensorMap fmap, const FgArgs g) {
  constexpr int K4 = kSpK - 1;               // float4 per row kept in shared memory
  constexpr int CS = L * K4 + 1;             // chunk stride (float4), padded
  constexpr int SG = SB / 8;                 // system groups of 8 per CTA
  constexpr int NG = L / 8;                  // 8-row groups per chunk
  const int M = g.M, P = g.P, batch = g.batch, T = g.T;
  const int nslot = P - (g.dup_hi - g.dup_lo);
  // the TMA destination (the tile at the start) must be 128-byte aligned
  extern __shared__ __align__(128) float4 smem4[];
  // [RS][SB] f tile (TMA), then the tables and the per-block scratch
  double* tile = reinterpret_cast<double*>(smem4);
  float4* rtab = smem4 + (TMA ? tile_bytes(g.RS, SB) / sizeof(float4) : 0);   // [nslot][CS]
  float2* ctab2 = reinterpret_cast<float2*>(rtab + (size_t)nslot * CS);      // [P][kSpChunk]
  float2* sE = ctab2 + (size_t)P * kSpChunk;                                 // [SB][P][2]
  float2* sW = sE + (size_t)SB * P * 2;                                      // [SB][P][2]
  uint32_t* smax = reinterpret_cast<uint32_t*>(sW + (size_t)SB * P * 2);     // [SB]
  __shared__ uint64_t bar;
  __shared__ int s_next;                     // the CTA's next block (thread 0 writes it after barrier 1)

  for (int t = threadIdx.x; t < P * L * K4; t += blockDim.x) {
    const int row = t / K4, k = t % K4, cc = row / L;
    if (cc > g.dup_lo && cc <= g.dup_hi) continue;                 // shares chunk dup_lo's slot
    cp_async16(&rtab[row_slot(cc, g.dup_lo, g.dup_hi) * CS + (row % L) * K4 + k],
               &g.rowtab[(size_t)row * kSpK + k]);
  }
  for (int t = threadIdx.x; t < P * kSpChunk / 2; t += blockDim.x)
    cp_async16(&ctab2[2 * t], &g.chunk_df[2 * t]);
  for (int t = threadIdx.x; t < SB; t += blockDim.x) smax[t] = 0u;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int sys = (w % SG) * 8 + (lane & 7);
  const int c = (w / SG) * 4 + (lane >> 3);
  const int row0 = c * L;
  const long long ld = batch;
  const int nblk = (batch + SB - 1) / SB;
  // the first block's tile: TMA boxes of SB systems x BR rows (rows past M and
  // systems past the batch arrive as zeros)
  if constexpr (TMA) {
    // a misaligned tile would fault the copy: report it and leave instead
    if ((tma::smem_u32(tile) & 127u) != 0u) {
      if (threadIdx.x == 0) atomicExch(g.err, 2);
      return;
    }
    if (threadIdx.x == 0) {
      tma::mbar_init(&bar, 1);
      if ((int)blockIdx.x < nblk) {
        tma::mbar_expect_tx(&bar, (unsigned)tile_bytes(g.RS, SB));
        for (int y = 0; y < g.RS; y += g.BR) tma::load_2d(tile + (size_t)y * SB, &fmap, blockIdx.x * SB, y, &bar);
      }
    }
  } else if (blockIdx.x * SB + sys < batch) {
    // the first block's rows start towards L2 while the tables arrive
    const double* pf = g.X + (long long)row0 * ld + blockIdx.x * SB + sys;
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (row0 + j < M) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf + (long long)j * ld));
  }
  cp_async_wait_all();
  __syncthreads();

  const float4* ctb = rtab + (size_t)row_slot(c, g.dup_lo, g.dup_hi) * CS;   // this chunk's rows
  const float2* ct = ctab2 + (size_t)c * kSpChunk;
  const float B = g.B;

  // Blocks after the first gridDim.x come from a queue (an atomic counter), so
  // CTAs that run faster take more of them: of the two CTAs sharing an SM the
  // warp scheduler favours one, which with a fixed share of the blocks finished
  // in 70% of the other's time, leaving the SM to one CTA (at under half the
  // two-CTA rate) for the rest of the launch.
  unsigned phase = 0;
  for (int blk = blockIdx.x; blk < nblk; phase ^= 1u) {
    const int s = blk * SB + sys;
    const bool act = s < batch;
    double* p = g.X + (long long)row0 * ld + (act ? s : 0);

    // ---- 1. load; the system's largest |f| sets its scale
    double fv[L];
    // the block after the next one is claimed now; the claim returns while the
    // tile is read, and its tile is requested after barrier 1
    unsigned claim = 0u;
    if (threadIdx.x == 0) claim = atomicAdd(&g.sched[0], 1u);
    bool tile_ok = true;
    if constexpr (TMA) {
      // bounded wait for the tile (2 s); the CTA agrees on the outcome at
      // barrier 1 (a thread whose wait failed reads stale data, which no one uses)
      tile_ok = tma::mbar_wait(&bar, phase, 2000000000ull);
      // Chunks start 2 KB apart, so the four chunks of a warp would read the
      // same 16 banks; odd chunks read each pair of rows in swapped order,
      // which puts them on the other 16 banks.
      const double* tr = tile + (size_t)row0 * SB + sys;
      const int sw = c & 1;
#pragma unroll
      for (int j = 0; j < L; j += 2) {
        const double u0 = tr[(j + sw) * SB], u1 = tr[(j + 1 - sw) * SB];
        fv[j] = sw ? u1 : u0;
        fv[j + 1] = sw ? u0 : u1;
      }
    } else {
#pragma unroll
      for (int j = 0; j < L; ++j) fv[j] = (act && row0 + j < M) ? p[j * ld] : 0.0;
    }
    uint32_t mx = 0u, nz = 0u;
#pragma unroll
    for (int j = 0; j < L; j += 2) mx = max(mx, fg::mag_pair(fv[j], fv[j + 1], nz));
    atomicMax(&smax[sys], mx | (nz != 0u ? 1u : 0u));
    // barrier 1: tile read, smax complete (the warps of the previous block are
    // all past its barrier 3, after which nothing reads what this block writes
    // before here)
    if (__syncthreads_or(!tile_ok)) {
      if (threadIdx.x == 0) atomicExch(g.err, 1);
      break;
    }
    if (threadIdx.x == 0) {
      const int nb = (int)gridDim.x + (int)claim;
      s_next = nb;
      // the next block's tile streams in behind the rest of this block
      if (TMA && nb < nblk) {
        tma::mbar_expect_tx(&bar, (unsigned)tile_bytes(g.RS, SB));
        for (int y = 0; y < g.RS; y += g.BR) tma::load_2d(tile + (size_t)y * SB, &fmap, nb * SB, y, &bar);
      }
    }
    const fg::SysClass sc = fg::classify(smax[sys], kEMin, kEMax);
    const bool native = act && !sc.fast && !sc.zero && !sc.resc;
    const uint32_t ioff = fg::in_offset(sc.ein), ooff = fg::out_offset(sc.eo);
    const bool zero = sc.zero, resc = sc.resc;
    const int dres = sc.d;

    // local forward sweep, zero incoming state: g_j = r f_j + P g_{j-2} + Q g_{j-1}
    float va[L], vl[L];
    {
      float y1h = 0.f, y1l = 0.f, y2h = 0.f, y2l = 0.f;
#pragma unroll
      for (int j = 0; j < L; ++j) {
        const float4 c0 = ctb[j * K4];
        const float4 c1 = ctb[j * K4 + 1];
        float fh, fl, a, l;
        fg::split(fv[j], ioff, fh, fl);
        fg::start(a, l, B, c0.x, c0.y, fh, fl);
        fg::madd(a, l, c0.z, c0.w, y2h, y2l);
        fg::madd(a, l, c1.x, c1.y, y1h, y1l);
        va[j] = a;
        vl[j] = l;
        y2h = y1h;
        y2l = y1l;
        y1h = __fsub_rn(a, B);
        y1l = l;
      }
    }
    {
      float2* eo2 = sE + ((size_t)sys * P + c) * 2;
      eo2[0] = make_float2(__fsub_rn(va[L - 2], B), vl[L - 2]);
      eo2[1] = make_float2(__fsub_rn(va[L - 1], B), vl[L - 1]);
    }
    // local back substitution, zero outgoing state: y_j = g_j + C y_{j+1} + D y_{j+2}
    {
      float x1h = 0.f, x1l = 0.f, x2h = 0.f, x2l = 0.f;
#pragma unroll
      for (int j = L - 1; j >= 0; --j) {
        const float4 c2 = ctb[j * K4 + 2];
        float a = va[j], l = vl[j];
        fg::madd(a, l, c2.z, c2.w, x2h, x2l);
        fg::madd(a, l, c2.x, c2.y, x1h, x1l);
        va[j] = a;
        vl[j] = l;
        x2h = x1h;
        x2l = x1l;
        x1h = __fsub_rn(a, B);
        x1l = l;
      }
    }

    // ---- 2. boundary states (truncated parallel scan), on the solve's grid: the
    // plan's bound covers them, and a fixed-grid multiply-add has a two-FMA
    // critical path where a TwoSum sum of products has about ten
    __syncthreads();                                     // e_c published, smax read
    if (c == 0) smax[sys] = 0u;                          // for the next block (ordered by the next barrier)
    D2 S0{0.f, 0.f}, S1{0.f, 0.f}, T0{0.f, 0.f}, T1{0.f, 0.f};
    {
      const float2* E = sE + (size_t)sys * P * 2;
      float s0a = B, s0l = 0.f, s1a = B, s1l = 0.f;      // biased accumulators
      for (int k = 1; k <= T && k <= c; ++k) {           // s_c = sum_k A_{c,k} e_{c-k}
        const float2 ea = E[2 * (c - k)], eb = E[2 * (c - k) + 1];
        if (k == 1) {
          s0a = __fadd_rn(s0a, ea.x); s0l = __fadd_rn(s0l, ea.y);
          s1a = __fadd_rn(s1a, eb.x); s1l = __fadd_rn(s1l, eb.y);
        } else {
          const float2* A = ct + 12 + 4 * (k - 2);
          fg::madd(s0a, s0l, A[0].x, A[0].y, ea.x, ea.y);
          fg::madd(s0a, s0l, A[1].x, A[1].y, eb.x, eb.y);
          fg::madd(s1a, s1l, A[2].x, A[2].y, ea.x, ea.y);
          fg::madd(s1a, s1l, A[3].x, A[3].y, eb.x, eb.y);
        }
      }
      S0 = D2{__fsub_rn(s0a, B), s0l};
      S1 = D2{__fsub_rn(s1a, B), s1l};
      // w_c = x'_start + Mst_c s_c
      float w0a = va[0], w0l = vl[0], w1a = va[1], w1l = vl[1];
      const float2* Ms = ct + 4;
      fg::madd(w0a, w0l, Ms[0].x, Ms[0].y, S0.h, S0.l);
      fg::madd(w0a, w0l, Ms[1].x, Ms[1].y, S1.h, S1.l);
      fg::madd(w1a, w1l, Ms[2].x, Ms[2].y, S0.h, S0.l);
      fg::madd(w1a, w1l, Ms[3].x, Ms[3].y, S1.h, S1.l);
      float2* wo = sW + ((size_t)sys * P + c) * 2;
      wo[0] = make_float2(__fsub_rn(w0a, B), w0l);
      wo[1] = make_float2(__fsub_rn(w1a, B), w1l);
    }
    __syncthreads();                                     // w_c published
    {
      const float2* Wv = sW + (size_t)sys * P * 2;
      float t0a = B, t0l = 0.f, t1a = B, t1l = 0.f;
      for (int k = 0; k < T && c + 1 + k < P; ++k) {     // t_c = sum_k B_{c,k} w_{c+1+k}
        const float2 wa = Wv[2 * (c + 1 + k)], wb = Wv[2 * (c + 1 + k) + 1];
        if (k == 0) {
          t0a = __fadd_rn(t0a, wa.x); t0l = __fadd_rn(t0l, wa.y);
          t1a = __fadd_rn(t1a, wb.x); t1l = __fadd_rn(t1l, wb.y);
        } else {
          const float2* Bk = ct + 24 + 4 * (k - 1);
          fg::madd(t0a, t0l, Bk[0].x, Bk[0].y, wa.x, wa.y);
          fg::madd(t0a, t0l, Bk[1].x, Bk[1].y, wb.x, wb.y);
          fg::madd(t1a, t1l, Bk[2].x, Bk[2].y, wa.x, wa.y);
          fg::madd(t1a, t1l, Bk[3].x, Bk[3].y, wb.x, wb.y);
        }
      }
      T0 = D2{__fsub_rn(t0a, B), t0l};
      T1 = D2{__fsub_rn(t1a, B), t1l};
    }

    // ---- 3. x = x' + M1 s0 + M2 s1 + K1 t0 + K2 t1, joined to fp64 and stored
    // an all-zero system already holds its solution (the solve is in place)
    const bool store = act && !native && !zero;
    // Three rows in four join through integer operations, the fourth through
    // one fp64 add: with every output on the fp64 pipe, that pipe (a warp
    // instruction per 64 cycles of a sub-partition) held the output phase.
    // Measured at N = 1024, batch 65536: all rows fp64 0.312 ms, one in four
    // through integers 0.300, two 0.302, three 0.298, all four 0.306.
    auto out = [&](const int j, const float h, const float l) {
      return (j & 3) != 0 ? fg::join_int(h, l, ooff) : fg::join(h, l, ooff);
    };
    // One 8-row group of corrections, join and store, with the kinds of its M
    // and K terms fixed (1 low word, 2 full): straight-line code.  The kinds
    // the plans produce are full/full in the middle of a chunk and full/low,
    // low/full near its ends; other groups test the kinds per row.
    auto group = [&](const int j0, auto mkind, auto kkind) {
      constexpr int MK = decltype(mkind)::value, KK = decltype(kkind)::value;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        float a = va[j], l = vl[j];
        if constexpr (MK > 0) {
          const float4 c3 = ctb[j * K4 + 3];
          if constexpr (MK == 2) {
            fg::madd(a, l, c3.x, c3.y, S0.h, S0.l);
            fg::madd(a, l, c3.z, c3.w, S1.h, S1.l);
          } else {
            fg::madd_low(l, c3.x, S0.h);
            fg::madd_low(l, c3.z, S1.h);
          }
        }
        if constexpr (KK > 0) {
          const float4 c4 = ctb[j * K4 + 4];
          if constexpr (KK == 2) {
            fg::madd(a, l, c4.x, c4.y, T0.h, T0.l);
            fg::madd(a, l, c4.z, c4.w, T1.h, T1.l);
          } else {
            fg::madd_low(l, c4.x, T0.h);
            fg::madd_low(l, c4.z, T1.h);
          }
        }
        fg::store_cs_if(p + j * ld, out(j, __fsub_rn(a, B), l), store && row0 + j < M);
      }
    };
    using K1 = std::integral_constant<int, 1>;
    using K2 = std::integral_constant<int, 2>;
    // one test per group picks its kinds (0 none, 1 low word, 2 full; the plan
    // fixed them per 8-row group)
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const int mk = gi < g.gm_full ? 2 : (gi < g.gm_none ? 1 : 0);
      const int kk = gi >= g.gk_full ? 2 : (gi >= g.gk_none ? 1 : 0);
      const int j0 = gi * 8;
      if (mk == 2 && kk == 2) {
        group(j0, K2{}, K2{});
      } else if (mk == 2 && kk == 1) {
        group(j0, K2{}, K1{});
      } else if (mk == 1 && kk == 2) {
        group(j0, K1{}, K2{});
      } else {
        // other kinds: tested per row
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + u;
          float a = va[j], l = vl[j];
          const float4 c3 = ctb[j * K4 + 3];
          const float4 c4 = ctb[j * K4 + 4];
          if (mk == 2) {
            fg::madd(a, l, c3.x, c3.y, S0.h, S0.l);
            fg::madd(a, l, c3.z, c3.w, S1.h, S1.l);
          } else if (mk == 1) {
            fg::madd_low(l, c3.x, S0.h);
            fg::madd_low(l, c3.z, S1.h);
          }
          if (kk == 2) {
            fg::madd(a, l, c4.x, c4.y, T0.h, T0.l);
            fg::madd(a, l, c4.z, c4.w, T1.h, T1.l);
          } else if (kk == 1) {
            fg::madd_low(l, c4.x, T0.h);
            fg::madd_low(l, c4.z, T1.h);
          }
          fg::store_cs_if(p + j * ld, out(j, __fsub_rn(a, B), l), store && row0 + j < M);
        }
      }
    }
    // rescaled systems: their stored rows are x * 2^(eo - e), scaled back here
    // (this thread's own stores, re-read in program order)
    if (act && resc) {
      const double post = fg::pow2i(dres);
      asm volatile("" ::: "memory");
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (row0 + j < M) p[j * ld] *= post;
    }
    // systems whose largest entry is subnormal or not finite: one thread solves
    // the column in fp64 (its f is untouched: nothing of it has been stored)
    if (native && c == 0) native_solve_col(NativeTabs{g.coef64, g.tail64, nullptr}, g.X + s, M, (size_t)ld, 0);
    blk = s_next;                                        // written before barrier 2
  }
  // the last CTA out leaves the queue at zero for the next launch (its claims,
  // and every other CTA's, precede their count)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&g.sched[1], 1u) == gridDim.x - 1u) {
      atomicExch(&g.sched[0], 0u);
      atomicExch(&g.sched[1], 0u);
    }
  }
}

size_t fg_smem_bytes(int L, int P, int SB, int nslot, int RS, bool with_tile) {
  const int K4 = kSpK - 1;
  return (with_tile ? tile_bytes(RS, SB) : 0) + (size_t)nslot * (L * K4 + 1) * sizeof(float4) +
         (size_t)P * kSpChunk * sizeof(float2) + 2 * (size_t)SB * P * 2 * sizeof(float2) +
         (size_t)SB * sizeof(uint32_t);
}

// rows per TMA box and staged rows for an M-row block
void tile_rows(int M, int& BR, int& RS) {
  BR = M <= 256 ? ((M + 7) & ~7) : 256;
  RS = (M + BR - 1) / BR * BR;
}

template <int L, int SB, int MAXT>
cudaError_t launch(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const int P = p.sp_P;
  const int nslot = P - (p.fg_dup_hi - p.fg_dup_lo);
  int BR = 0, RS = 0;
  tile_rows(p.M, BR, RS);
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  const size_t smem_tile = fg_smem_bytes(L, P, SB, nslot, RS, true);
  const bool tma = RS >= L * P && smem_tile <= kStepsSmemMax &&
                   tma::encode_2d(&map, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, sizeof(double), batch, p.M,
                                  (unsigned)SB, (unsigned)BR);
  const size_t smem = tma ? smem_tile : fg_smem_bytes(L, P, SB, nslot, RS, false);
  auto kern = tma ? k_fg<L, SB, MAXT, true> : k_fg<L, SB, MAXT, false>;
  const int nblk = (batch + SB - 1) / SB;
  int per_sm = 0;
  const cudaError_t e = kernel_prepare((const void*)kern, smem, SB * P, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  int grid = per_sm * p.num_sms;
  if (grid > nblk) grid = nblk;
  FgArgs a;
  a.rowtab = p.sptab;
  a.chunk_df = p.spchunk_df;
  a.coef64 = p.coef64;
  a.tail64 = p.tail64;
  a.X = X;
  a.err = p.kern_err;
  a.sched = p.sched;
  a.M = p.M;
  a.P = P;
  a.batch = batch;
  a.T = p.sp_T;
  a.dup_lo = p.fg_dup_lo;
  a.dup_hi = p.fg_dup_hi;
  a.RS = RS;
  a.BR = BR;
  a.B = p.fg_bias;
  a.gm_full = p.fg_gm_full;
  a.gm_none = p.fg_gm_none;
  a.gk_none = p.fg_gk_none;
  a.gk_full = p.fg_gk_full;
  kern<<<grid, SB * P, smem, st>>>(map, a);
  note_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// plan time: bounds on the solve's intermediate values and the grid
// ---------------------------------------------------------------------------

// Largest row sum of |L^-1 R| (g = L^-1 R f: the forward substitution's
// operator) and of |A^-1|, from the native fp64 tables.  Each column's
// impulse response is propagated until its two-term state is below 2^-80 of
// its start (the recurrences of a nonsingular banded factor decay), or to the
// end of the block.
void inverse_row_sums(const std::vector<double>& cf, int M, double& Gg, double& Gx) {
  const double* R = cf.data() + (size_t)kR * M;
  const double* P = cf.data() + (size_t)kP * M;
  const double* Q = cf.data() + (size_t)kQ * M;
  const double* G = cf.data() + (size_t)kGam * M;
  const double* D = cf.data() + (size_t)kDel * M;
  std::vector<double> rg(M, 0.0), rx(M, 0.0), gcol(M, 0.0);
  for (int k = 0; k < M; ++k) {
    const double tiny = std::ldexp(std::fabs(R[k]), -80);
    int end = k;
    double g1 = 0.0, g2 = 0.0;
    for (int i = k; i < M; ++i) {
      const double gi = (i == k ? R[k] : 0.0) - P[i] * g2 - Q[i] * g1;
      gcol[i] = gi;
      rg[i] += std::fabs(gi);
      g2 = g1;
      g1 = gi;
      end = i;
      if (i > k + 1 && std::fabs(g1) < tiny && std::fabs(g2) < tiny) break;
    }
    double x1 = 0.0, x2 = 0.0;
    double xmax = 0.0;
    for (int i = end; i >= 0; --i) {
      const double xi = (i >= k ? gcol[i] : 0.0) - G[i] * x1 - D[i] * x2;
      rx[i] += std::fabs(xi);
      xmax = std::max(xmax, std::fabs(xi));
      x2 = x1;
      x1 = xi;
      if (i < k - 1 && std::fabs(x1) < 1e-24 * xmax && std::fabs(x2) < 1e-24 * xmax) break;
    }
  }
  Gg = *std::max_element(rg.begin(), rg.end());
  Gx = *std::max_element(rx.begin(), rx.end());
}

}  // namespace

// Decide whether the plan's partitioned solves can run on a fixed grid and
// set the grid and the correction-term groups.  Needs the partitioned tables
// (L = 32, truncated chunk scan, non-cyclic) and the native tables on the
// device; up to 64 chunks the one-CTA kernel runs on it (fg_ok), beyond that
// the local sweeps and the fix-up of the long-system kernels (big_fg).
cudaError_t fg_prepare(pent_plan_s& p) {
  p.fg_ok = 0;
  p.big_fg = 0;
  if (p.cyclic || p.sp_L != 32 || p.sp_T <= 0) return cudaSuccess;
  const int M = p.M, L = p.sp_L, P = p.sp_P, Mpad = L * P;
  // up to 64 chunks: the one-CTA kernel (k_fg); beyond: the grid for the
  // kernels of systems too long for one CTA
  const bool one_cta = P <= 64;
  std::vector<double> cf((size_t)kCoefCount * M);
  std::vector<float4> rows((size_t)Mpad * kSpK);
  cudaError_t e = cudaMemcpy(cf.data(), p.coef64, cf.size() * sizeof(double), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(rows.data(), p.sptab, rows.size() * sizeof(float4), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  // longest run of chunks whose kernel row tables (kSpK - 1 float4 per row) are
  // bitwise equal to the run's first: they share one shared-memory slot
  if (one_cta) {
    const int K4 = kSpK - 1;
    auto same = [&](int a, int b) {
      for (int j = 0; j < L; ++j)
        if (std::memcmp(&rows[((size_t)a * L + j) * kSpK], &rows[((size_t)b * L + j) * kSpK],
                        K4 * sizeof(float4)) != 0)
          return false;
      return true;
    };
    int best_lo = 0, best_hi = 0;
    for (int c = 1; c < P;) {
      if (!same(c - 1, c)) { ++c; continue; }
      const int lo = c - 1;
      while (c < P && same(lo, c)) ++c;
      if (c - 1 - lo > best_hi - best_lo) { best_lo = lo; best_hi = c - 1; }
    }
    p.fg_dup_lo = best_lo;
    p.fg_dup_hi = best_hi;
  }
  if (one_cta) {
    int BR = 0, RS = 0;
    tile_rows(M, BR, RS);
    const int nslot = P - (p.fg_dup_hi - p.fg_dup_lo);
    if (fg_smem_bytes(L, P, 8, nslot, RS, false) > kStepsSmemMax) return cudaSuccess;
  }
  double Gg = 0.0, Gx = 0.0;
  inverse_row_sums(cf, M, Gg, Gx);
  auto val = [&](int row, int k, int half) {
    const float4 q = rows[(size_t)row * kSpK + k];
    return half ? (double)q.z + (double)q.w : (double)q.x + (double)q.y;
  };
  // Bound on every partial sum for max |f| = 1: forward rows (|r| + (|P| + |Q|) Gg),
  // the local back substitution (its chunk-local |R^-1| row sums times Gg), and
  // the corrections (|x'| + (|M1| + |M2|) Gg + (|K1| + |K2|) Gx).
  double bound = std::max(Gg, Gx);
  std::vector<double> mM(L, 0.0), mK(L, 0.0);
  for (int c = 0; c < P; ++c) {
    // chunk-local row sums of the back substitution's inverse
    std::vector<double> us(L, 0.0);
    for (int k = 0; k < L; ++k) {
      double x1 = 0.0, x2 = 0.0;
      for (int j = k; j >= 0; --j) {
        const int row = c * L + j;
        const double xj = (j == k ? 1.0 : 0.0) + val(row, 2, 0) * x1 + val(row, 2, 1) * x2;
        us[j] += std::fabs(xj);
        x2 = x1;
        x1 = xj;
      }
    }
    const double Gu = *std::max_element(us.begin(), us.end());
    for (int j = 0; j < L; ++j) {
      const int row = c * L + j;
      const double fwd = std::fabs(val(row, 0, 0)) + (std::fabs(val(row, 0, 1)) + std::fabs(val(row, 1, 0))) * Gg;
      const double bwd = Gg + (std::fabs(val(row, 2, 0)) + std::fabs(val(row, 2, 1))) * Gu * Gg;
      const double m = std::fabs(val(row, 3, 0)) + std::fabs(val(row, 3, 1));
      const double kk = std::fabs(val(row, 4, 0)) + std::fabs(val(row, 4, 1));
      const double cor = Gu * Gg + m * Gg + kk * Gx;
      bound = std::max(bound, std::max(fwd, std::max(bwd, cor)));
      mM[j] = std::max(mM[j], std::max(std::fabs(val(row, 3, 0)), std::fabs(val(row, 3, 1))));
      mK[j] = std::max(mK[j], std::max(std::fabs(val(row, 4, 0)), std::fabs(val(row, 4, 1))));
    }
  }
  if (!(bound > 0.0) || !std::isfinite(bound) || bound > 64.0) return cudaSuccess;
  // max |f| < 2 after scaling, and a margin for the low words: every partial sum
  // below 2^(k+22)
  const int kexp = (int)std::ceil(std::log2(2.5 * bound)) - 22;
  p.fg_bias = std::ldexp(1.5f, kexp + 23);
  // correction groups: full while any response in the group is >= 2^-24,
  // low word while >= 2^-56, none after (M decays down a chunk, K up it)
  const int NG = L / 8;
  auto gmax = [&](const std::vector<double>& v, int gi) {
    double m = 0.0;
    for (int j = 8 * gi; j < 8 * gi + 8; ++j) m = std::max(m, v[j]);
    return m;
  };
  int gm_full = 0, gm_none = 0;
  for (int gi = 0; gi < NG; ++gi) {
    if (gmax(mM, gi) >= std::ldexp(1.0, -24)) gm_full = gi + 1;
    if (gmax(mM, gi) >= std::ldexp(1.0, -56)) gm_none = gi + 1;
  }
  int gk_full = NG, gk_none = NG;
  for (int gi = NG - 1; gi >= 0; --gi) {
    if (gmax(mK, gi) >= std::ldexp(1.0, -24)) gk_full = gi;
    if (gmax(mK, gi) >= std::ldexp(1.0, -56)) gk_none = gi;
  }
  p.fg_gm_full = gm_full;
  p.fg_gm_none = std::max(gm_none, gm_full);
  p.fg_gk_full = gk_full;
  p.fg_gk_none = std::min(gk_none, gk_full);
  p.fg_bound = bound;
  if (one_cta) p.fg_ok = 1;
  else p.big_fg = 1;
  return cudaSuccess;
}

cudaError_t shared_fg(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  return p.sp_P <= 32 ? launch<32, 8, 256>(p, X, batch, st) : launch<32, 8, 512>(p, X, batch, st);
}

}  // namespace pent

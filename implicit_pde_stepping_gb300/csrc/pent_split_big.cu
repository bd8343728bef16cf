// Partitioned double-float solve for systems too long for one CTA.
//
// The mathematics of pent_split_df.cu (cuPentBatch's forward substitution
// L g = f and back substitution R x = g per chunk of L rows, chunk boundary
// states s_c, t_c by the truncated chunk-coupling scan, Navon's bordering,
// eqs. (8)–(12), for periodic plans), split over kernels because a system's
// P chunks no longer fit in one CTA:
//   k_big_local   one thread per (system, chunk): load f, local forward and back
//                 substitution with zero boundary states; x' (double-float pair,
//                 8 bytes) goes back in place of f; summaries e_c (local forward
//                 end values) and x'_start(c) go to a small array;
//   k_big_states  one thread per (system, chunk): s_c = sum_k A_{c,k} e_{c-k},
//                 w_c = x'_start(c) + Mst_c s_c;
//   k_big_border  periodic plans, one thread per system: t at chunk 0 and at the
//                 chunks holding rows M-2, M-1, y at rows 0, 1, M-2, M-1 and
//                 x_t = S^{-1}(f_t - H^T y), written to rows M, M+1;
//   k_big_fix     one thread per (system, chunk): t_c = sum_k B_{c,k} w_{c+1+k},
//                 x = x' + M1 s0 + M2 s1 + K1 t0 + K2 t1 (- U x_t), stored in fp64.
// Range: every chunk converts its rows with its own power of two (the one that
// puts its largest |entry| in [1, 2), known from the rows it loads; a chunk
// whose largest entry is subnormal is first multiplied by 2^600 in fp64, which
// is exact), so the pairs' float exponent range never limits a chunk.  Each
// chunk records its exponent, and k_big_local folds two words per system into
// global memory with one atomic per CTA: the largest magnitude (a system with an
// inf or NaN entry returns NaN everywhere; an all-zero one is left as it is, its
// own solution) and the largest chunk exponent E.  k_big_states and k_big_fix
// bring each chunk's pairs to the system's scale 2^E by exact power-of-two
// multiplications (terms more than 2^-126 below the system's largest value are
// flushed), and k_big_fix joins the result to fp64 at 2^E, or for E outside the
// window of the integer conversion at the window's edge followed by one fp64
// multiplication.
// Memory traffic: f read once (k_big_local), x' written and read, x written,
// plus summaries of 64 bytes and one exponent per chunk.  The chunk states are
// computed in double-float like the sweeps (summaries and a copy of the chunk
// tables as (hi, lo) pairs), which keeps them off the fp64 pipe; only the
// periodic border (one thread per system) works in fp64.  The parallelism is
// batch x P threads, so a handful of very long systems still fills the GPU.
#include <type_traits>

#include "cp_async.cuh"
#include "df64.cuh"
#include "fg.cuh"
#include "pent_internal.cuh"

namespace pent {
namespace {

using df::D2;

constexpr int kBigL = 32;       // rows per chunk (the plan's sp_L for long systems)

// Chunk whose tables chunk c uses: chunks dup.x < c <= dup.y have tables
// bitwise equal to chunk dup.x's (found when the plan was built), so they all
// read those, which stay in cache.
__device__ __forceinline__ int table_chunk(int c, int2 dup) { return (c > dup.x && c <= dup.y) ? dup.x : c; }
constexpr int kBigThreads = 256;
// threads of k_big_local and k_big_fix: CTAs of 4 warps, each staging its rows in
// 32 KB of shared memory, four CTAs to an SM (0.164 -> 0.161 ms per solve of 16
// systems of 2^20 rows against CTAs of 8 warps, two to an SM)
constexpr int kLocalThreads = 128;
constexpr int kSum = 8;         // doubles per (chunk, system): e(2) x'start(2) s(2) w(2)

__device__ __forceinline__ void mv2(const double* A, double x0, double x1, double& y0, double& y1) {
  y0 = fma(A[0], x0, fma(A[1], x1, y0));
  y1 = fma(A[2], x0, fma(A[3], x1, y1));
}

// (system, chunk) of this thread: SPW consecutive systems per warp row, so a
// load instruction covers SPW * 8 bytes of each of 32 / SPW rows.  The grid's x
// runs over groups of systems and y over groups of chunks, so the CTAs that
// read the same table rows for different systems are scheduled together and
// share them through L2.
template <int SPW, int NT>
__device__ __forceinline__ void place(int& s, int& c) {
  constexpr int CPW = 32 / SPW;                      // chunks per warp
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  s = blockIdx.x * SPW + lane % SPW;
  c = (blockIdx.y * (NT / 32) + w) * CPW + lane / SPW;
}

constexpr int kZeroChunk = -(1 << 20);   // chunk exponent of an all-zero (or non-finite) chunk
constexpr int kExpBias = 1024;           // the per-system exponent word holds E + kExpBias (0: none)

// x 2^d for |d| up to about 2000: two exact power-of-two products (only the
// last can round, where the result is subnormal)
__device__ __forceinline__ double scale2(double x, int d) {
  const int d1 = d / 2;
  return (x * fg::pow2i(d1)) * fg::pow2i(d - d1);
}

// 2^d as a float for d <= 0, flushed to 0 below 2^-126
__device__ __forceinline__ float pow2f(int d) { return d >= -126 ? __uint_as_float((uint32_t)(127 + d) << 23) : 0.f; }
__device__ __forceinline__ D2 scaled(D2 v, float f) { return D2{v.h * f, v.l * f}; }

// Magnitude word of n values at a stride of kLocalThreads doubles (a separate
// call, so that the sweeps that follow reload f instead of keeping it live)
__device__ __noinline__ uint32_t column_word(const double* v, int n) {
  uint32_t mx = 0u, nz = 0u;
  for (int j = 0; j < n; ++j) {
    const double f = v[j * kLocalThreads];
    mx = max(mx, fg::mag_bits(f));
    nz |= (uint32_t)__double2loint(f);
  }
  return mx | (nz != 0u ? 1u : 0u);
}

// One thread per (system, chunk): the chunk's exponent from its own rows, the
// local sweeps in that scale, x' in place of f, the summaries, and the two
// per-system words (largest magnitude, largest chunk exponent), reduced over
// the CTA and folded in with one atomic each (both zeroed before).
template <int SPW, bool CYC, bool FG>
__global__ void __launch_bounds__(kLocalThreads, 4)
    k_big_local(const float4* __restrict__ tab, double* __restrict__ X, double* __restrict__ sum,
                double* __restrict__ xm, unsigned* __restrict__ smag, unsigned* __restrict__ sexp,
                int* __restrict__ cexp, int M, int P, int batch, int2 dup, float B) {
  constexpr int L = kBigL;
  constexpr int NT = kLocalThreads;
  constexpr int NW = NT / 32;
  __shared__ unsigned red[2][NW][SPW];
  int s, c;
  place<SPW, NT>(s, c);
  const bool act = s < batch && c < P;
  const long long ld = batch;
  const int row0 = c * L;
  double* p = X + (long long)row0 * ld + (act ? s : 0);
  // the chunk's f into this thread's shared-memory column, every row in flight at once
  extern __shared__ double sf[];                  // [L][NT]
  double* mine = sf + threadIdx.x;
  if (act) {
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (row0 + j < M) cp_async8(mine + j * NT, p + (long long)j * ld);
  }
  cp_async_wait_all();
  // magnitude word: largest high word without sign, bit 0 set if any low word is nonzero
  const uint32_t mword = act ? column_word(mine, row0 + L <= M ? L : M - row0) : 0u;
  const uint32_t mx = mword & ~1u;
  int ce = kZeroChunk;                            // the chunk's exponent: pairs = f 2^-(ce - 1023)
  uint32_t econv = 1023u;                         // exponent field the conversion rebiases by
  if (mword != 0u && (mx >> 20) != 0x7FFu) {
    if ((mx >> 20) == 0u) {
      // largest entry subnormal: the chunk times 2^600 first (exact), so that the
      // integer conversion reads normal numbers
      uint32_t m2 = 0u;
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (row0 + j < M) {
          const double f = mine[j * NT] * 0x1p600;
          mine[j * NT] = f;
          m2 = max(m2, fg::mag_bits(f));
        }
      econv = m2 >> 20;
      ce = (int)econv - 600;
    } else {
      econv = mx >> 20;
      ce = (int)econv;
    }
  }
  // per-system words over the CTA (its warps share the same SPW systems), one
  // atomic each per CTA and system
  {
    uint32_t a = act ? mword : 0u, b = (act && ce != kZeroChunk) ? (uint32_t)(ce + kExpBias) : 0u;
#pragma unroll
    for (int o = SPW; o < 32; o <<= 1) {
      a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane < SPW) {
      red[0][w][lane] = a;
      red[1][w][lane] = b;
    }
    __syncthreads();
    if (threadIdx.x < SPW && blockIdx.x * SPW + (int)threadIdx.x < batch) {
      uint32_t ma = 0u, mb = 0u;
#pragma unroll
      for (int k = 0; k < NW; ++k) {
        ma = max(ma, red[0][k][threadIdx.x]);
        mb = max(mb, red[1][k][threadIdx.x]);
      }
      if (ma) atomicMax(smag + blockIdx.x * SPW + threadIdx.x, ma);
      if (mb) atomicMax(sexp + blockIdx.x * SPW + threadIdx.x, mb);
    }
  }
  if (!act) return;
  cexp[(size_t)c * batch + s] = ce;
  float2* o = reinterpret_cast<float2*>(sum) + ((size_t)c * batch + s) * kSum;
  if (ce == kZeroChunk) {
    // all zero (already its own x') or not finite (the system returns NaN)
    o[0] = o[1] = o[2] = o[3] = make_float2(0.f, 0.f);
    if (CYC) {
#pragma unroll
      for (int j = 0; j < L; ++j) {
        if (row0 + j == M - 2) xm[(size_t)s * 2] = 0.0;
        if (row0 + j == M - 1) xm[(size_t)s * 2 + 1] = 0.0;
      }
    }
    return;
  }
  const uint32_t off = fg::in_offset(econv);
  const float4* t = tab + (size_t)table_chunk(c, dup) * L * kSpK;
  D2 v[L];
  if constexpr (FG) {
    // the sweeps on the plan's fixed grid (pent_fg.cu, fg.cuh): bias B, values
    // (a - B) + l; the plan bounds them for a chunk whose largest |f| is in [1, 2)
    float va[L], vl[L];
    {
      float y1h = 0.f, y1l = 0.f, y2h = 0.f, y2l = 0.f;
#pragma unroll
      for (int j = 0; j < L; ++j) {
        const double f = (row0 + j < M) ? mine[j * NT] : 0.0;
        const float4 c0 = __ldg(t + j * kSpK), c1 = __ldg(t + j * kSpK + 1);
        float fh, fl, a, l;
        fg::split(f, off, fh, fl);
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
    o[0] = make_float2(__fsub_rn(va[L - 2], B), vl[L - 2]);
    o[1] = make_float2(__fsub_rn(va[L - 1], B), vl[L - 1]);
    {
      float x1h = 0.f, x1l = 0.f, x2h = 0.f, x2l = 0.f;
#pragma unroll
      for (int j = L - 1; j >= 0; --j) {
        const float4 c2 = __ldg(t + j * kSpK + 2);
        float a = va[j], l = vl[j];
        fg::madd(a, l, c2.z, c2.w, x2h, x2l);
        fg::madd(a, l, c2.x, c2.y, x1h, x1l);
        x2h = x1h;
        x2l = x1l;
        x1h = __fsub_rn(a, B);
        x1l = l;
        v[j] = D2{x1h, l};
      }
    }
  } else {
    {
      D2 a1{0.f, 0.f}, a2{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < L; ++j) {
        const double f = (row0 + j < M) ? mine[j * NT] : 0.0;
        const float4 c0 = __ldg(t + j * kSpK), c1 = __ldg(t + j * kSpK + 1);
        float fh, fl;
        fg::split(f, off, fh, fl);
        const D2 g = df::sum3p(D2{c0.x, c0.y}, D2{fh, fl}, D2{c0.z, c0.w}, a2, D2{c1.x, c1.y}, a1);
        v[j] = g;
        a2 = a1;
        a1 = g;
      }
    }
    o[0] = make_float2(v[L - 2].h, v[L - 2].l);
    o[1] = make_float2(v[L - 1].h, v[L - 1].l);
    {
      D2 a1{0.f, 0.f}, a2{0.f, 0.f};
#pragma unroll
      for (int j = L - 1; j >= 0; --j) {
        const float4 c2 = __ldg(t + j * kSpK + 2);
        const D2 y = df::sum3(v[j], D2{c2.x, c2.y}, a1, D2{c2.z, c2.w}, a2);
        v[j] = y;
        a2 = a1;
        a1 = y;
      }
    }
  }
  o[2] = make_float2(v[0].h, v[0].l);
  o[3] = make_float2(v[1].h, v[1].l);
  if (CYC) {                                      // x' at rows M-2, M-1 for the border, in the chunk's scale
#pragma unroll
    for (int j = 0; j < L; ++j) {
      if (row0 + j == M - 2) xm[(size_t)s * 2] = df::to_double(v[j]);
      if (row0 + j == M - 1) xm[(size_t)s * 2 + 1] = df::to_double(v[j]);
    }
  }
  float2* q = reinterpret_cast<float2*>(p);       // x' in place of f, as (hi, lo), in the chunk's scale
#pragma unroll
  for (int j = 0; j < L; ++j)
    if (row0 + j < M) q[j * ld] = make_float2(v[j].h, v[j].l);
}

__device__ __forceinline__ D2 d2(float2 v) { return D2{v.x, v.y}; }
__device__ __forceinline__ float2 f2(D2 v) { return make_float2(v.h, v.l); }

// y += A x for a row-major 2x2 A, double-float
__device__ __forceinline__ void mv2d(const float2* A, D2 x0, D2 x1, D2& y0, D2& y1) {
  y0 = df::sum3(y0, d2(A[0]), x0, d2(A[1]), x1);
  y1 = df::sum3(y1, d2(A[2]), x0, d2(A[3]), x1);
}

// The system's exponent E (the largest chunk exponent) from its two words:
// false for an all-zero system (nothing to do) and a non-finite one.
__device__ __forceinline__ bool system_exp(const unsigned* smag, const unsigned* sexp, int s, int& E) {
  const unsigned mag = smag[s], ew = sexp[s];
  E = (int)ew - kExpBias;
  return ew != 0u && (mag >> 20) != 0x7FFu;
}

// s_c from the local end values of the T chunks before c (summaries as (hi, lo),
// each in its own chunk's scale, brought to the system's scale 2^E)
__device__ __forceinline__ void state_s(const float2* __restrict__ ctab, const float2* __restrict__ sum,
                                        const int* __restrict__ cexp, int c, int s, int batch, int T, int2 dup,
                                        int E, D2& s0, D2& s1) {
  const float2* ct = ctab + (size_t)table_chunk(c, dup) * kSpChunk;
  s0 = s1 = D2{0.f, 0.f};
  for (int k = 1; k <= T && k <= c; ++k) {
    const size_t i = (size_t)(c - k) * batch + s;
    const float2* e = sum + i * kSum;
    const float f = pow2f(cexp[i] - E);
    const D2 ea = scaled(d2(e[0]), f), eb = scaled(d2(e[1]), f);
    if (k == 1) { s0 = df::add(s0, ea); s1 = df::add(s1, eb); }
    else mv2d(ct + 12 + 4 * (k - 2), ea, eb, s0, s1);
  }
}

// t_c from w of the T chunks after c (already in the system's scale)
__device__ __forceinline__ void state_t(const float2* __restrict__ ctab, const float2* __restrict__ sum,
                                        int c, int s, int P, int batch, int T, int2 dup, D2& t0, D2& t1) {
  const float2* ct = ctab + (size_t)table_chunk(c, dup) * kSpChunk;
  t0 = t1 = D2{0.f, 0.f};
  for (int k = 0; k < T && c + 1 + k < P; ++k) {
    const float2* w = sum + ((size_t)(c + 1 + k) * batch + s) * kSum + 6;
    if (k == 0) { t0 = df::add(t0, d2(w[0])); t1 = df::add(t1, d2(w[1])); }
    else mv2d(ct + 24 + 4 * (k - 1), d2(w[0]), d2(w[1]), t0, t1);
  }
}

__global__ void __launch_bounds__(kBigThreads)
    k_big_states(const float2* __restrict__ ctab, const double* __restrict__ extra, float2* __restrict__ sum,
                 const unsigned* __restrict__ smag, const unsigned* __restrict__ sexp,
                 const int* __restrict__ cexp, int P, int batch, int2 dup) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)P * batch) return;
  const int c = (int)(i / batch), s = (int)(i % batch);
  int E;
  if (!system_exp(smag, sexp, s, E)) return;
  const int T = (int)extra[18];
  D2 s0, s1;
  state_s(ctab, sum, cexp, c, s, batch, T, dup, E, s0, s1);
  float2* o = sum + (size_t)i * kSum;
  const float f = pow2f(cexp[i] - E);
  D2 w0 = scaled(d2(o[2]), f), w1 = scaled(d2(o[3]), f);
  mv2d(ctab + (size_t)table_chunk(c, dup) * kSpChunk + 4, s0, s1, w0, w1);   // w_c = x'_start + Mst_c s_c
  o[4] = f2(s0);
  o[5] = f2(s1);
  o[6] = f2(w0);
  o[7] = f2(w1);
}

// the chunk tables as double-float pairs (plan time)
__global__ void k_chunk_df(const double* __restrict__ src, float2* __restrict__ dst, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = f2(df::from_double(src[i]));
}

__global__ void __launch_bounds__(kBigThreads)
    k_big_border(const double* __restrict__ ctab, const float2* __restrict__ ctabd,
                 const double* __restrict__ extra, const float2* __restrict__ sum,
                 const double* __restrict__ xm, double* __restrict__ X, const unsigned* __restrict__ smag,
                 const unsigned* __restrict__ sexp, const int* __restrict__ cexp, int M, int P, int batch,
                 int2 dup) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  int E;
  if (!system_exp(smag, sexp, s, E)) return;
  const long long ld = batch;
  const int T = (int)extra[18];
  // y at rows 0, 1: chunk 0 has s_0 = 0, so y = w_0 + Kst_0 t_0
  D2 td0, td1;
  state_t(ctabd, sum, 0, s, P, batch, T, dup, td0, td1);
  const float2* o0 = sum + (size_t)s * kSum;
  double y0 = df::to_double(d2(o0[6])), y1 = df::to_double(d2(o0[7]));
  mv2(ctab + 8, df::to_double(td0), df::to_double(td1), y0, y1);
  // y at rows M-2, M-1 from their chunks' x' (in the chunk's scale), s and t
  double yv[2];
  for (int r = 0; r < 2; ++r) {
    const int row = M - 2 + r, c = row / kBigL;
    const float2* oc = sum + ((size_t)c * batch + s) * kSum;
    D2 u0, u1;
    state_t(ctabd, sum, c, s, P, batch, T, dup, u0, u1);
    const double* mk = extra + 10 + 2 * r;   // M1, M2 at the row; K1, K2 four slots on
    yv[r] = scale2(xm[(size_t)s * 2 + r], cexp[(size_t)c * batch + s] - E) + mk[0] * df::to_double(d2(oc[4])) +
            mk[1] * df::to_double(d2(oc[5])) + mk[4] * df::to_double(u0) + mk[5] * df::to_double(u1);
  }
  const double r0 = extra[4] * yv[0] + extra[5] * yv[1] + extra[6] * y0;
  const double r1 = extra[7] * yv[1] + extra[8] * y0 + extra[9] * y1;
  // in the system's scale; the border solution back at its own scale
  const double f0 = scale2(X[(long long)M * ld + s], 1023 - E), f1 = scale2(X[(long long)(M + 1) * ld + s], 1023 - E);
  X[(long long)M * ld + s] = scale2(extra[0] * (f0 - r0) + extra[1] * (f1 - r1), E - 1023);
  X[(long long)(M + 1) * ld + s] = scale2(extra[2] * (f0 - r0) + extra[3] * (f1 - r1), E - 1023);
}

// cold paths of k_big_fix, out of line
__device__ __noinline__ void fill_nan(double* p, long long ld, int n) {
  for (int j = 0; j < n; ++j) p[j * ld] = __longlong_as_double(0x7FF8000000000000ll);
}
__device__ __noinline__ void scale_rows(double* p, long long ld, int n, double f) {
  for (int j = 0; j < n; ++j) p[j * ld] *= f;
}

template <int SPW, bool CYC, bool FG>
__global__ void __launch_bounds__(kLocalThreads, 4)
    k_big_fix(const float4* __restrict__ tab, const float2* __restrict__ ctab,
              const double* __restrict__ extra, const float2* __restrict__ sum, double* __restrict__ X,
              const unsigned* __restrict__ smag, const unsigned* __restrict__ sexp,
              const int* __restrict__ cexp, int M, int P, int batch, int2 dup, float B, int4 groups) {
  constexpr int L = kBigL;
  constexpr int NT = kLocalThreads;
  int s, c;
  place<SPW, NT>(s, c);
  if (s >= batch || c >= P) return;
  const long long ld = batch;
  const int row0 = c * L;
  if (row0 >= M) return;
  double* p = X + (long long)row0 * ld + s;
  const int nrow = M - row0 < L ? M - row0 : L;
  if (sexp[s] != 0u && (smag[s] >> 20) == 0x7FFu) {
    // an inf or NaN entry: the system's solution is not finite
    fill_nan(p, ld, nrow);
    if (CYC && c == 0) fill_nan(X + (long long)M * ld + s, ld, 2);
    return;
  }
  int E;
  if (!system_exp(smag, sexp, s, E)) return;      // all zero: already solved
  // the chunk's x' (pairs) into this thread's shared-memory column, every row in
  // flight while the chunk states are formed
  extern __shared__ float2 sx[];                  // [L][NT]
  float2* mine = sx + threadIdx.x;
  const float2* q = reinterpret_cast<const float2*>(p);
#pragma unroll
  for (int j = 0; j < L; ++j)
    if (j < nrow) cp_async8(mine + j * NT, q + (long long)j * ld);
  // the join to fp64 at 2^E, or at the edge of its window and then one fp64 product
  const int eo = E < (int)fg::kEMin ? (int)fg::kEMin : (E > (int)fg::kEMax ? (int)fg::kEMax : E);
  const uint32_t off = fg::out_offset((uint32_t)eo);
  const float fx = pow2f(cexp[(size_t)c * batch + s] - E);   // x' from the chunk's scale to the system's
  const int T = (int)extra[18];
  const float2* o = sum + ((size_t)c * batch + s) * kSum;
  D2 T0, T1;
  state_t(ctab, sum, c, s, P, batch, T, dup, T0, T1);
  const D2 S0 = d2(o[4]), S1 = d2(o[5]);
  bool needU = false;
  D2 X0{0.f, 0.f}, X1{0.f, 0.f};
  if (CYC) {
    const int reach = (int)extra[19];
    needU = c < reach || c > (M - 1) / L - reach;
    X0 = df::from_double(-scale2(X[(long long)M * ld + s], 1023 - E));
    X1 = df::from_double(-scale2(X[(long long)(M + 1) * ld + s], 1023 - E));
  }
  cp_async_wait_all();
  const float4* t = tab + (size_t)table_chunk(c, dup) * L * kSpK;
  auto emit = [&](int j, D2 x) {
    // three rows in four join through integers, off the slow fp64 pipe
    const double xo = (j & 3) != 0 ? fg::join_int(x.h, x.l, off) : fg::join(x.h, x.l, off);
    fg::store_cs_if(p + j * ld, xo, j < nrow);
  };
  if constexpr (FG) {
    // on the plan's grid: x' (brought to the system's scale) onto it exactly, then
    // the correction terms as fixed-grid multiply-adds, in 8-row groups whose kinds
    // the plan fixed (2 full, 1 low word alone, 0 none; the M responses fall down a
    // chunk, the K responses up it); one row with the kinds of its terms
    // (compile-time in the common groups, tested per row in the others)
    auto row = [&](int j, auto mk, auto kk) {
      const float2 xv = j < nrow ? mine[j * NT] : make_float2(0.f, 0.f);
      const float hs = xv.x * fx, ls = xv.y * fx;
      float a = __fadd_rn(B, hs);
      float l = __fadd_rn(ls, __fsub_rn(hs, __fsub_rn(a, B)));
      const float4 c3 = __ldg(t + j * kSpK + 3), c4 = __ldg(t + j * kSpK + 4);
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
      emit(j, D2{__fsub_rn(a, B), l});
    };
    using K1 = std::integral_constant<int, 1>;
    using K2 = std::integral_constant<int, 2>;
#pragma unroll
    for (int gi = 0; gi < L / 8; ++gi) {
      const int mk = gi < groups.x ? 2 : (gi < groups.y ? 1 : 0);
      const int kk = gi >= groups.w ? 2 : (gi >= groups.z ? 1 : 0);
      const int j0 = gi * 8;
      if (mk == 2 && kk == 2) {
#pragma unroll
        for (int u = 0; u < 8; ++u) row(j0 + u, K2{}, K2{});
      } else if (mk == 2 && kk == 1) {
#pragma unroll
        for (int u = 0; u < 8; ++u) row(j0 + u, K2{}, K1{});
      } else if (mk == 1 && kk == 2) {
#pragma unroll
        for (int u = 0; u < 8; ++u) row(j0 + u, K1{}, K2{});
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) row(j0 + u, mk, kk);
      }
    }
  } else {
#pragma unroll 8
    for (int j = 0; j < L; ++j) {
      const float2 xv = j < nrow ? mine[j * NT] : make_float2(0.f, 0.f);
      const float4 c3 = __ldg(t + j * kSpK + 3), c4 = __ldg(t + j * kSpK + 4);
      D2 x = df::axpy(scaled(D2{xv.x, xv.y}, fx), D2{c3.x, c3.y}, S0);
      x = df::axpy(x, D2{c3.z, c3.w}, S1);
      x = df::axpy(x, D2{c4.x, c4.y}, T0);
      x = df::axpy(x, D2{c4.z, c4.w}, T1);
      if (CYC && needU) {
        const float4 c1 = __ldg(t + j * kSpK + 1), c5 = __ldg(t + j * kSpK + 5);
        x = df::axpy(x, D2{c1.z, c1.w}, X0);
        x = df::axpy(x, D2{c5.x, c5.y}, X1);
      }
      emit(j, x);
    }
  }
  if (eo != E) {
    // outside the join's window: the stored rows are x 2^(eo - E), scaled back
    // (this thread's own stores, re-read in program order)
    asm volatile("" ::: "memory");
    scale_rows(p, ld, M - row0 < L ? M - row0 : L, fg::pow2i(E - eo));
  }
}

template <int SPW, bool CYC>
cudaError_t run(pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const int P = p.sp_P;
  constexpr int CPB = (kLocalThreads / 32) * (32 / SPW);   // chunks per CTA
  const dim3 grid((batch + SPW - 1) / SPW, (P + CPB - 1) / CPB);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  // scratch: summaries, x' at rows M-2, M-1, the two per-system words, chunk exponents
  double* xm = p.spsum + (size_t)P * batch * kSum;
  unsigned* smag = reinterpret_cast<unsigned*>(xm + 2 * (size_t)batch);
  unsigned* sexp = smag + batch;
  int* cexp = reinterpret_cast<int*>(sexp + batch);
  const int2 dup = make_int2(p.dup_lo, p.dup_hi);
  const size_t smem_local = (size_t)kBigL * kLocalThreads * sizeof(double);
  const size_t smem_fix = (size_t)kBigL * kLocalThreads * sizeof(float2);
  // non-cyclic plans whose grid the plan derived: sweeps and fix-up on it
  const bool fgrid = !CYC && p.big_fg && p.fg_use;
  auto local = fgrid ? k_big_local<SPW, CYC, true> : k_big_local<SPW, CYC, false>;
  auto fix = fgrid ? k_big_fix<SPW, CYC, true> : k_big_fix<SPW, CYC, false>;
  cudaError_t e = kernel_prepare((const void*)local, smem_local, kLocalThreads, nullptr);
  if (e == cudaSuccess) e = kernel_prepare((const void*)fix, smem_fix, kLocalThreads, nullptr);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(smag, 0, 2 * (size_t)batch * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  local<<<grid, kLocalThreads, smem_local, st>>>(p.sptab, X, p.spsum, xm, smag, sexp, cexp, p.M, P, batch, dup,
                                               p.fg_bias);
  note_launch();
  const long long n = (long long)P * batch;
  float2* sumd = reinterpret_cast<float2*>(p.spsum);
  k_big_states<<<(unsigned)((n + kBigThreads - 1) / kBigThreads), kBigThreads, 0, st>>>(
      p.spchunk_df, p.spextra, sumd, smag, sexp, cexp, P, batch, dup);
  note_launch();
  if (CYC) {
    k_big_border<<<(batch + kBigThreads - 1) / kBigThreads, kBigThreads, 0, st>>>(
        p.spchunk, p.spchunk_df, p.spextra, sumd, xm, X, smag, sexp, cexp, p.M, P, batch, dup);
    note_launch();
  }
  // correction groups of the grid kernels (the TwoSum form applies every term)
  const int4 groups = make_int4(p.fg_gm_full, p.fg_gm_none, p.fg_gk_none, p.fg_gk_full);
  fix<<<grid, kLocalThreads, smem_fix, st>>>(p.sptab, p.spchunk_df, p.spextra, sumd, X, smag, sexp, cexp, p.M, P,
                                             batch, dup, p.fg_bias, groups);
  note_launch();
  return cudaGetLastError();
}

template <bool CYC>
cudaError_t run_cyc(pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  if (batch >= 8) return run<8, CYC>(p, X, batch, st);
  if (batch >= 4) return run<4, CYC>(p, X, batch, st);
  if (batch >= 2) return run<2, CYC>(p, X, batch, st);
  return run<1, CYC>(p, X, batch, st);
}

}  // namespace

cudaError_t split_big_prepare(pent_plan_s& p, cudaStream_t st) {
  const int n = p.sp_P * kSpChunk;
  k_chunk_df<<<(n + 255) / 256, 256, 0, st>>>(p.spchunk, p.spchunk_df, n);
  note_launch();
  return cudaGetLastError();
}

cudaError_t shared_split_big(pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  if (p.sp_L != kBigL || p.sp_T <= 0) return cudaErrorInvalidValue;
  // summaries: kSum doubles per (chunk, system), then x' at rows M-2, M-1 per
  // system, two words per system, one exponent per (chunk, system)
  const size_t need = ((size_t)p.sp_P * batch * kSum + 2 * (size_t)batch) * sizeof(double) +
                      2 * (size_t)batch * sizeof(unsigned) + (size_t)p.sp_P * batch * sizeof(int);
  if (p.spsum_bytes < need) {
    if (p.spsum) {
      cudaError_t e = cudaStreamSynchronize(st);   // earlier solves may still read it
      if (e != cudaSuccess) return e;
      cudaFree(p.spsum);
      p.spsum = nullptr;
      p.spsum_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&p.spsum, need);
    if (e != cudaSuccess) return e;
    p.spsum_bytes = need;
  }
  return p.cyclic ? run_cyc<true>(p, X, batch, st) : run_cyc<false>(p, X, batch, st);
}

}  // namespace pent

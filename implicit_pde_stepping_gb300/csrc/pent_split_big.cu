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
// Range: a first kernel (k_big_scale) takes each system's largest |entry|, and
// the others work on the system scaled by the power of two that puts it in
// [1, 2) (folded into the fp64 <-> pair conversions), so the pairs' float
// exponent range never limits the result; a system outside the scaled path's
// window (largest entry zero, subnormal, non-finite or extreme) is left
// untouched by the first kernels and solved natively in fp64 by one thread of
// k_big_fix.
// Memory traffic: f read twice (the scale pass and k_big_local), x' written
// and read, x written, plus summaries of 64 bytes per chunk.  The chunk states are
// computed in double-float like the sweeps (summaries and a copy of the chunk
// tables as (hi, lo) pairs), which keeps them off the fp64 pipe; only the
// periodic border (one thread per system) works in fp64.  The parallelism is
// batch x P threads, so a handful of very long systems still fills the GPU.
#include "cp_async.cuh"
#include "df64.cuh"
#include "fg.cuh"
#include "pent_internal.cuh"
#include "pent_native.cuh"

namespace pent {
namespace {

using df::D2;

constexpr int kBigL = 32;       // rows per chunk (the plan's sp_L for long systems)

// Chunk whose tables chunk c uses: chunks dup.x < c <= dup.y have tables
// bitwise equal to chunk dup.x's (found when the plan was built), so they all
// read those, which stay in cache.
__device__ __forceinline__ int table_chunk(int c, int2 dup) { return (c > dup.x && c <= dup.y) ? dup.x : c; }
constexpr int kBigThreads = 256;
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
template <int SPW>
__device__ __forceinline__ void place(int& s, int& c) {
  constexpr int CPW = 32 / SPW;                      // chunks per warp
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  s = blockIdx.x * SPW + lane % SPW;
  c = (blockIdx.y * (kBigThreads / 32) + w) * CPW + lane / SPW;
}

// the system's exponent window check (largest-entry exponent field e)
__device__ __forceinline__ bool big_fast(uint32_t e) { return e >= fg::kEMin && e <= fg::kEMax; }

// largest |entry| of each system (rows 0..N-1): SPW systems per warp row, the
// rows strided over the grid; lanes of one system, then the CTA's warps reduce,
// and one atomic per CTA and system combines into smax[s] (zeroed before).
// The word is the largest fp64 high word without sign, with bit 0 set if any
// low word is nonzero: 0 marks an all-zero system, which the other kernels
// leave untouched (zero is its solution, in place).
template <int SPW>
__global__ void __launch_bounds__(kBigThreads)
    k_big_scale(const double* __restrict__ X, unsigned* __restrict__ smax, int rows, int batch) {
  constexpr int RPW = 32 / SPW;                   // rows per warp and step
  constexpr int NW = kBigThreads / 32;
  __shared__ unsigned red[NW][SPW];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int s = blockIdx.x * SPW + lane % SPW;
  unsigned mx = 0u, nz = 0u;
  if (s < batch) {
    const long long ld = batch;
    const int stride = gridDim.y * NW * RPW;
#pragma unroll 8
    for (int i = (blockIdx.y * NW + w) * RPW + lane / SPW; i < rows; i += stride) {
      const double v = X[(long long)i * ld + s];
      mx = max(mx, fg::mag_bits(v));
      nz |= (uint32_t)__double2loint(v);
    }
  }
  mx |= nz != 0u ? 1u : 0u;                       // only an all-zero system ends at 0
#pragma unroll
  for (int o = SPW; o < 32; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane < SPW) red[w][lane] = mx;
  __syncthreads();
  if (threadIdx.x < SPW && blockIdx.x * SPW + (int)threadIdx.x < batch) {
    unsigned m = 0u;
#pragma unroll
    for (int k = 0; k < NW; ++k) m = max(m, red[k][threadIdx.x]);
    atomicMax(smax + blockIdx.x * SPW + threadIdx.x, m);
  }
}

template <int SPW, bool CYC>
__global__ void __launch_bounds__(kBigThreads, 2)
    k_big_local(const float4* __restrict__ tab, double* __restrict__ X, double* __restrict__ sum,
                double* __restrict__ xm, const unsigned* __restrict__ smax, int M, int P, int batch,
                int2 dup) {
  constexpr int L = kBigL;
  int s, c;
  place<SPW>(s, c);
  if (s >= batch || c >= P) return;
  if (smax[s] == 0u) return;                      // all zero: already solved
  const uint32_t e = smax[s] >> 20;
  if (!big_fast(e)) return;                       // solved natively by k_big_fix
  const uint32_t off = fg::in_offset(e);
  const long long ld = batch;
  const int row0 = c * L;
  double* p = X + (long long)row0 * ld + s;
  const float4* t = tab + (size_t)table_chunk(c, dup) * L * kSpK;
  // the chunk's f into this thread's shared-memory column, every row in flight at once
  extern __shared__ double sf[];                  // [L][kBigThreads]
  double* mine = sf + threadIdx.x;
#pragma unroll
  for (int j = 0; j < L; ++j)
    if (row0 + j < M) cp_async8(mine + j * kBigThreads, p + (long long)j * ld);
  cp_async_wait_all();
  D2 v[L];
  {
    D2 a1{0.f, 0.f}, a2{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const double f = (row0 + j < M) ? mine[j * kBigThreads] : 0.0;
      const float4 c0 = __ldg(t + j * kSpK), c1 = __ldg(t + j * kSpK + 1);
      float fh, fl;
      fg::split(f, off, fh, fl);
      const D2 g = df::sum3p(D2{c0.x, c0.y}, D2{fh, fl}, D2{c0.z, c0.w}, a2, D2{c1.x, c1.y}, a1);
      v[j] = g;
      a2 = a1;
      a1 = g;
    }
  }
  float2* o = reinterpret_cast<float2*>(sum) + ((size_t)c * batch + s) * kSum;
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
  o[2] = make_float2(v[0].h, v[0].l);
  o[3] = make_float2(v[1].h, v[1].l);
  if (CYC) {                                      // x' at rows M-2, M-1 for the border
#pragma unroll
    for (int j = 0; j < L; ++j) {
      if (row0 + j == M - 2) xm[(size_t)s * 2] = df::to_double(v[j]);
      if (row0 + j == M - 1) xm[(size_t)s * 2 + 1] = df::to_double(v[j]);
    }
  }
  float2* q = reinterpret_cast<float2*>(p);       // x' in place of f, as (hi, lo)
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

// s_c from the local end values of the T chunks before c (summaries as (hi, lo))
__device__ __forceinline__ void state_s(const float2* __restrict__ ctab, const float2* __restrict__ sum,
                                        int c, int s, int batch, int T, int2 dup, D2& s0, D2& s1) {
  const float2* ct = ctab + (size_t)table_chunk(c, dup) * kSpChunk;
  s0 = s1 = D2{0.f, 0.f};
  for (int k = 1; k <= T && k <= c; ++k) {
    const float2* e = sum + ((size_t)(c - k) * batch + s) * kSum;
    if (k == 1) { s0 = df::add(s0, d2(e[0])); s1 = df::add(s1, d2(e[1])); }
    else mv2d(ct + 12 + 4 * (k - 2), d2(e[0]), d2(e[1]), s0, s1);
  }
}

// t_c from w of the T chunks after c
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
                 int P, int batch, int2 dup) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)P * batch) return;
  const int c = (int)(i / batch), s = (int)(i % batch);
  const int T = (int)extra[18];
  D2 s0, s1;
  state_s(ctab, sum, c, s, batch, T, dup, s0, s1);
  float2* o = sum + (size_t)i * kSum;
  D2 w0 = d2(o[2]), w1 = d2(o[3]);
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
                 const double* __restrict__ xm, double* __restrict__ X, const unsigned* __restrict__ smax,
                 int M, int P, int batch, int2 dup) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  if (smax[s] == 0u) return;                      // all zero: already solved
  const uint32_t e = smax[s] >> 20;
  if (!big_fast(e)) return;                       // solved natively by k_big_fix
  const long long ld = batch;
  const int T = (int)extra[18];
  // y at rows 0, 1: chunk 0 has s_0 = 0, so y = w_0 + Kst_0 t_0
  D2 td0, td1;
  state_t(ctabd, sum, 0, s, P, batch, T, dup, td0, td1);
  const float2* o0 = sum + (size_t)s * kSum;
  double y0 = df::to_double(d2(o0[6])), y1 = df::to_double(d2(o0[7]));
  mv2(ctab + 8, df::to_double(td0), df::to_double(td1), y0, y1);
  // y at rows M-2, M-1 from their chunks' s and t
  double yv[2];
  for (int r = 0; r < 2; ++r) {
    const int row = M - 2 + r, c = row / kBigL;
    const float2* oc = sum + ((size_t)c * batch + s) * kSum;
    D2 u0, u1;
    state_t(ctabd, sum, c, s, P, batch, T, dup, u0, u1);
    const double* mk = extra + 10 + 2 * r;   // M1, M2 at the row; K1, K2 four slots on
    yv[r] = xm[(size_t)s * 2 + r] + mk[0] * df::to_double(d2(oc[4])) + mk[1] * df::to_double(d2(oc[5])) +
            mk[4] * df::to_double(u0) + mk[5] * df::to_double(u1);
  }
  const double r0 = extra[4] * yv[0] + extra[5] * yv[1] + extra[6] * y0;
  const double r1 = extra[7] * yv[1] + extra[8] * y0 + extra[9] * y1;
  // in the system's scale; the border solution back at its own scale
  const double f0 = X[(long long)M * ld + s] * fg::pow2_neg(e), f1 = X[(long long)(M + 1) * ld + s] * fg::pow2_neg(e);
  X[(long long)M * ld + s] = (extra[0] * (f0 - r0) + extra[1] * (f1 - r1)) * fg::pow2_pos(e);
  X[(long long)(M + 1) * ld + s] = (extra[2] * (f0 - r0) + extra[3] * (f1 - r1)) * fg::pow2_pos(e);
}

template <int SPW, bool CYC>
__global__ void __launch_bounds__(kBigThreads)
    k_big_fix(const float4* __restrict__ tab, const float2* __restrict__ ctab,
              const double* __restrict__ extra, const float2* __restrict__ sum, double* __restrict__ X,
              const unsigned* __restrict__ smax, const NativeTabs nt, int M, int P, int batch, int2 dup) {
  constexpr int L = kBigL;
  int s, c;
  place<SPW>(s, c);
  if (s >= batch || c >= P) return;
  const long long ld = batch;
  if (smax[s] == 0u) return;                      // all zero: already solved
  const uint32_t e = smax[s] >> 20;
  if (!big_fast(e)) {                             // the whole column, natively, by one thread
    if (c == 0) native_solve_col(nt, X + s, M, (size_t)ld, CYC ? 1 : 0);
    return;
  }
  const uint32_t off = fg::in_offset(e);
  const int row0 = c * L;
  if (row0 >= M) return;
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
    X0 = df::from_double(-X[(long long)M * ld + s] * fg::pow2_neg(e));
    X1 = df::from_double(-X[(long long)(M + 1) * ld + s] * fg::pow2_neg(e));
  }
  double* p = X + (long long)row0 * ld + s;
  const float2* q = reinterpret_cast<const float2*>(p);
  const float4* t = tab + (size_t)table_chunk(c, dup) * L * kSpK;
  constexpr int G = 8;
#pragma unroll
  for (int j0 = 0; j0 < L; j0 += G) {
    float2 xv[G];
#pragma unroll
    for (int u = 0; u < G; ++u) xv[u] = (row0 + j0 + u < M) ? q[(j0 + u) * ld] : make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const int j = j0 + u;
      const float4 c3 = __ldg(t + j * kSpK + 3), c4 = __ldg(t + j * kSpK + 4);
      D2 x = df::axpy(D2{xv[u].x, xv[u].y}, D2{c3.x, c3.y}, S0);
      x = df::axpy(x, D2{c3.z, c3.w}, S1);
      x = df::axpy(x, D2{c4.x, c4.y}, T0);
      x = df::axpy(x, D2{c4.z, c4.w}, T1);
      if (CYC && needU) {
        const float4 c1 = __ldg(t + j * kSpK + 1), c5 = __ldg(t + j * kSpK + 5);
        x = df::axpy(x, D2{c1.z, c1.w}, X0);
        x = df::axpy(x, D2{c5.x, c5.y}, X1);
      }
      // three rows in four join through integers, off the slow fp64 pipe
      const double xo = (j & 3) != 0 ? fg::join_int(x.h, x.l, off) : fg::join(x.h, x.l, off);
      fg::store_cs_if(p + j * ld, xo, row0 + j < M);
    }
  }
}

template <int SPW, bool CYC>
cudaError_t run(pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const int P = p.sp_P;
  constexpr int CPB = (kBigThreads / 32) * (32 / SPW);     // chunks per CTA
  const dim3 grid((batch + SPW - 1) / SPW, (P + CPB - 1) / CPB);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  double* xm = p.spsum + (size_t)P * batch * kSum;
  unsigned* smax = reinterpret_cast<unsigned*>(xm + 2 * (size_t)batch);
  const int2 dup = make_int2(p.dup_lo, p.dup_hi);
  const size_t smem_local = (size_t)kBigL * kBigThreads * sizeof(double);
  cudaError_t e = kernel_prepare((const void*)k_big_local<SPW, CYC>, smem_local, kBigThreads, nullptr);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(smax, 0, (size_t)batch * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  {
    // enough CTAs over the rows to fill the GPU (each loops over its rows)
    const int rows = p.M + (CYC ? 2 : 0);
    const unsigned gx = (batch + SPW - 1) / SPW;
    const int per_cta = (kBigThreads / 32) * (32 / SPW);
    unsigned gy = (unsigned)((rows + per_cta - 1) / per_cta);
    const unsigned cap = (unsigned)(8 * (p.num_sms > 0 ? p.num_sms : 1)) / gx + 1;
    if (gy > cap) gy = cap;
    if (gy > 65535u) gy = 65535u;
    k_big_scale<SPW><<<dim3(gx, gy), kBigThreads, 0, st>>>(X, smax, rows, batch);
    note_launch();
  }
  k_big_local<SPW, CYC><<<grid, kBigThreads, smem_local, st>>>(p.sptab, X, p.spsum, xm, smax, p.M, P, batch,
                                                               dup);
  note_launch();
  const long long n = (long long)P * batch;
  float2* sumd = reinterpret_cast<float2*>(p.spsum);
  k_big_states<<<(unsigned)((n + kBigThreads - 1) / kBigThreads), kBigThreads, 0, st>>>(
      p.spchunk_df, p.spextra, sumd, P, batch, dup);
  note_launch();
  if (CYC) {
    k_big_border<<<(batch + kBigThreads - 1) / kBigThreads, kBigThreads, 0, st>>>(
        p.spchunk, p.spchunk_df, p.spextra, sumd, xm, X, smax, p.M, P, batch, dup);
    note_launch();
  }
  const NativeTabs nt{p.coef64, p.tail64, p.bands};
  k_big_fix<SPW, CYC><<<grid, kBigThreads, 0, st>>>(p.sptab, p.spchunk_df, p.spextra, sumd, X, smax, nt, p.M,
                                                   P, batch, dup);
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
  // system, then each system's largest |entry| bits
  const size_t need = ((size_t)p.sp_P * batch * kSum + 2 * (size_t)batch) * sizeof(double) +
                      (size_t)batch * sizeof(unsigned);
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

// Per-system pentadiagonal matrices, fp32: partitioned factor + solve with
// the CTA's tile loaded by TMA and the systems kept in registers.
//
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs" solves each
// system with one thread (the Rewrite variant: factorisation steps 1–14 and
// the two substitutions), which makes the factor coefficients gamma_i,
// delta_i and the intermediate g_i round-trip through memory.  Here a system is
// cut into P chunks of L = 16 rows, one thread per chunk, and its rows never
// leave the SM: memory sees the minimum (the five bands and f read once, x
// written once).
//
// Row i of the matrix: a_i x_{i-2} + b_i x_{i-1} + c_i x_i + d_i x_{i+1}
// + e_i x_{i+2} = f_i.  For the chunk of rows [s, e] write u = (x_{s-2},
// x_{s-1}) for the previous chunk's last two unknowns and v = (x_{e-1}, x_e)
// for its own.
//   1. Downward elimination (the page's factorisation, with the two unknowns
//      u carried as left spikes):
//          x_i + gamma_i x_{i+1} + delta_i x_{i+2} + p_i u0 + q_i u1 = g_i.
//      Two virtual rows x_{s-2} = u0, x_{s-1} = u1 start the recurrence, so
//      rows s and s+1 need no special case.
//   2. Upward elimination from row e-2 with v as the right unknowns:
//          x_i = Y_i - P_i u0 - Q_i u1 - R_i v0 - S_i v1.
//   3. The downward forms of rows e-1 and e reach into the next chunk's first
//      two rows, which are in form 2 with (v, v') in place of (u, v); that
//      leaves two equations per chunk in the t_c = v of chunk c:
//          Sub_c t_{c-1} + Dia_c t_c + Sup_c t_{c+1} = r_c,
//      a block tridiagonal system with 2x2 blocks, solved by parallel cyclic
//      reduction over P lanes with warp shuffles (each block row normalised
//      by its diagonal block first, so that a step exchanges 10 values).
//   4. Every row from form 2 with t_{c-1} and t_c.
// Layouts: interleaved [N][batch] (element (i, s) at i * batch + s), or
// block-interleaved with blocks of bs systems, each block an interleaved
// [N][bs] array: (i, s) at (s / bs) N bs + i bs + s % bs ("Simulating the
// behavior of the human brain on GPUs", section 4.1.1).  The TMA path loads a
// block-interleaved tile with 3-D tensor maps (bs a multiple of 16).
// No pivoting, as on the page (diagonally dominant or SPD matrices).  The
// chunk-local pivots are checked, and the first row whose pivot is zero or not
// finite is reported; failing that, the last row of the first chunk whose 2x2
// block in the reduced system is singular or not finite.
#include <climits>

#include "cp_async.cuh"
#include "pent_internal.cuh"
#include "tma.cuh"

namespace pent {
namespace {

constexpr int kSB = 16;   // systems per CTA
constexpr int kL = 16;    // rows per chunk

struct PsMaps {
  CUtensorMap m[6];   // a, b, c, d, e, f
};

__device__ __forceinline__ bool bad_pivot(float d) { return !(d != 0.f) || !isfinite(d); }
// fast reciprocal (about 1 ulp; the fp32 solve's tolerance is far wider)
__device__ __forceinline__ float rcp(float x) { return __fdividef(1.f, x); }

// 2x2 blocks, row-major {m00, m01, m10, m11}
struct M2 {
  float a, b, c, d;
};
__device__ __forceinline__ M2 mul(const M2& x, const M2& y) {
  return {fmaf(x.a, y.a, x.b * y.c), fmaf(x.a, y.b, x.b * y.d), fmaf(x.c, y.a, x.d * y.c),
          fmaf(x.c, y.b, x.d * y.d)};
}
__device__ __forceinline__ float2 mul(const M2& x, float2 v) {
  return {fmaf(x.a, v.x, x.b * v.y), fmaf(x.c, v.x, x.d * v.y)};
}
// inverse of m; ok is cleared if m is singular or not finite
__device__ __forceinline__ M2 inv(const M2& m, bool& ok) {
  const float det = fmaf(m.a, m.d, -m.b * m.c);
  if (bad_pivot(det)) ok = false;
  const float r = rcp(det);
  return {m.d * r, -m.b * r, -m.c * r, m.a * r};
}
__device__ __forceinline__ M2 shfl_up(const M2& m, int d, int w) {
  return {__shfl_up_sync(0xffffffffu, m.a, d, w), __shfl_up_sync(0xffffffffu, m.b, d, w),
          __shfl_up_sync(0xffffffffu, m.c, d, w), __shfl_up_sync(0xffffffffu, m.d, d, w)};
}
__device__ __forceinline__ M2 shfl_down(const M2& m, int d, int w) {
  return {__shfl_down_sync(0xffffffffu, m.a, d, w), __shfl_down_sync(0xffffffffu, m.b, d, w),
          __shfl_down_sync(0xffffffffu, m.c, d, w), __shfl_down_sync(0xffffffffu, m.d, d, w)};
}

// Interface data per chunk (20 values): the downward forms of its last two
// rows (gamma, delta, p, q, g at e-1, then at e) and the upward forms of its
// first two rows (Y, P, Q, R, S at s, then at s+1).
constexpr int kIface = 20;

// Dynamic shared memory: the staged tile (TMA: [6][RS rows][SB systems];
// cp.async: [6][L rows][SB * P threads]).  Once every thread has read its
// rows, the same space holds the interface data [20][P][SB + 1] and the
// chunk-end unknowns [2][P][SB + 1] (rows of SB + 1 so that both thread
// mappings, threads over systems and threads over chunks, spread over the banks).
template <int P, bool TMA>
__global__ void __launch_bounds__(kSB * P, P <= 16 ? 2 : 1)
    k_persys_split(const __grid_constant__ PsMaps maps, const float* __restrict__ A,
                   const float* __restrict__ B, const float* __restrict__ C, const float* __restrict__ D,
                   const float* __restrict__ E, float* __restrict__ X, int N, int batch, int bs, int RS,
                   int BR, int* __restrict__ info) {
  constexpr int SB = kSB, L = kL, NT = SB * P;
  extern __shared__ __align__(128) float smem[];
  float* const stage = smem;
  float (*const sI)[P][SB + 1] = reinterpret_cast<float (*)[P][SB + 1]>(smem);
  float (*const sT)[P][SB + 1] = reinterpret_cast<float (*)[P][SB + 1]>(smem + kIface * P * (SB + 1));
  __shared__ int sBad[SB];    // first bad chunk-local pivot (row, 1-based) per system
  __shared__ int sBadR[SB];   // first chunk-end row whose reduced-system block failed
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  const int lane = tid % SB;     // phases 1, 2, 4: system of this thread
  const int c = tid / SB;        //                 its chunk
  const int s = blockIdx.x * SB + lane;
  const bool act = s < batch;
  const size_t ld = bs ? (size_t)bs : (size_t)batch;                          // row stride
  const size_t sb = bs ? (size_t)(s / bs) * N * bs + s % bs : (size_t)s;     // row 0 of system s
  const int row0 = c * L;
  if (tid < SB) sBad[tid] = sBadR[tid] = INT_MAX;

  int bad = 0;
  // ---- 0. the tile into shared memory, all of it in flight at once
  if constexpr (TMA) {
    if (tid == 0) tma::mbar_init(&bar, 1);
    __syncthreads();
    if (tid == 0) {
      tma::mbar_expect_tx(&bar, (unsigned)(6 * RS * SB * sizeof(float)));
      for (int arr = 0; arr < 6; ++arr)
        for (int y0 = 0; y0 < RS; y0 += BR)
          if (bs)
            tma::load_3d(stage + ((size_t)arr * RS + y0) * SB, &maps.m[arr], (blockIdx.x * SB) % bs, y0,
                         (blockIdx.x * SB) / bs, &bar);
          else
            tma::load_2d(stage + ((size_t)arr * RS + y0) * SB, &maps.m[arr], blockIdx.x * SB, y0, &bar);
    }
    if (!tma::mbar_wait(&bar, 0, 2000000000ull)) bad = -1;   // 2 s: the copy never arrived
  } else {
    const float* src[6] = {A, B, C, D, E, X};
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const int i = row0 + j;
      if (act && i < N) {
        const size_t o = (size_t)i * ld + sb;
#pragma unroll
        for (int arr = 0; arr < 6; ++arr) cp_async4(&stage[(arr * L + j) * NT + tid], src[arr] + o);
      }
    }
    cp_async_wait_all();
  }
  auto staged = [&](int arr, int j) -> float {
    return TMA ? stage[((size_t)arr * RS + row0 + j) * SB + lane] : stage[(arr * L + j) * NT + tid];
  };

  // ---- 1. downward elimination with the left spikes p, q
  float gm[L], dl[L], pp[L], qq[L], gg[L];
  {
    // (gamma, delta, p, q, g) of rows j-2 and j-1, starting from the virtual rows
    // x_{s-2} - u0 = 0 and x_{s-1} - u1 = 0
    float g2 = 0.f, g1 = 0.f, d2 = 0.f, d1 = 0.f, p2 = -1.f, p1 = 0.f, q2 = 0.f, q1 = -1.f, y2 = 0.f,
          y1 = 0.f;
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const int i = row0 + j;
      const bool in = act && i < N;
      const float a = (in && i >= 2) ? staged(0, j) : 0.f;
      const float b = (in && i >= 1) ? staged(1, j) : 0.f;
      const float cc = in ? staged(2, j) : 1.f;
      const float d = (in && i + 1 < N) ? staged(3, j) : 0.f;
      const float e = (in && i + 2 < N) ? staged(4, j) : 0.f;
      const float f = in ? staged(5, j) : 0.f;
      const float beta = fmaf(-a, g2, b);
      const float alpha = fmaf(-beta, g1, fmaf(-a, d2, cc));
      if (bad == 0 && bad_pivot(alpha)) bad = i + 1;
      const float ra = rcp(alpha);
      gm[j] = fmaf(-beta, d1, d) * ra;
      dl[j] = e * ra;
      pp[j] = -fmaf(a, p2, beta * p1) * ra;
      qq[j] = -fmaf(a, q2, beta * q1) * ra;
      gg[j] = fmaf(-beta, y1, fmaf(-a, y2, f)) * ra;
      g2 = g1; g1 = gm[j];
      d2 = d1; d1 = dl[j];
      p2 = p1; p1 = pp[j];
      q2 = q1; q1 = qq[j];
      y2 = y1; y1 = gg[j];
    }
  }
  // downward forms of rows e-1 (A) and e (B), for the reduced system
  const float gA = gm[L - 2], dA = dl[L - 2], pA = pp[L - 2], qA = qq[L - 2], yA = gg[L - 2];
  const float gB = gm[L - 1], dB = dl[L - 1], pB = pp[L - 1], qB = qq[L - 1], yB = gg[L - 1];

  // ---- 2. upward elimination, in place: Y in gg, P in pp, Q in qq, R in gm, S in dl.
  //      Rows e-1 and e take the trivial forms x = v0 and x = v1.
  gg[L - 2] = gg[L - 1] = 0.f;
  pp[L - 2] = pp[L - 1] = 0.f;
  qq[L - 2] = qq[L - 1] = 0.f;
  gm[L - 2] = -1.f; dl[L - 2] = 0.f;
  gm[L - 1] = 0.f;  dl[L - 1] = -1.f;
#pragma unroll
  for (int j = L - 3; j >= 0; --j) {
    const float gj = gm[j], dj = dl[j];
    gg[j] = fmaf(-gj, gg[j + 1], fmaf(-dj, gg[j + 2], gg[j]));
    pp[j] = fmaf(-gj, pp[j + 1], fmaf(-dj, pp[j + 2], pp[j]));
    qq[j] = fmaf(-gj, qq[j + 1], fmaf(-dj, qq[j + 2], qq[j]));
    gm[j] = -fmaf(gj, gm[j + 1], dj * gm[j + 2]);
    dl[j] = -fmaf(gj, dl[j + 1], dj * dl[j + 2]);
  }

  __syncthreads();   // every thread has read its rows of the tile: its space is free
  {
    const float w[kIface] = {gA, dA, pA, qA, yA, gB, dB, pB, qB, yB,
                             gg[0], pp[0], qq[0], gm[0], dl[0], gg[1], pp[1], qq[1], gm[1], dl[1]};
#pragma unroll
    for (int k = 0; k < kIface; ++k) sI[k][c][lane] = w[k];
  }
  if (bad) atomicMin(&sBad[lane], bad);
  __syncthreads();

  // ---- 3. chunk-end unknowns: block tridiagonal system per system, PCR over P lanes
  {
    const int q = tid / P;   // system of this lane group
    const int k = tid % P;   // its chunk
    const bool last = k == P - 1;
    const float a_g = sI[0][k][q], a_d = sI[1][k][q], a_p = sI[2][k][q], a_q = sI[3][k][q], a_y = sI[4][k][q];
    const float b_g = sI[5][k][q], b_d = sI[6][k][q], b_p = sI[7][k][q], b_q = sI[8][k][q], b_y = sI[9][k][q];
    float n[10];
#pragma unroll
    for (int m = 0; m < 10; ++m) n[m] = last ? 0.f : sI[10 + m][k + 1][q];
    // next chunk's rows s', s'+1: x = Yn - Pn v0 - Qn v1 - Rn w0 - Sn w1
    const float Y0 = n[0], P0 = n[1], Q0 = n[2], R0 = n[3], S0 = n[4];
    const float Y1 = n[5], P1 = n[6], Q1 = n[7], R1 = n[8], S1 = n[9];
    const M2 sub = k > 0 ? M2{a_p, a_q, b_p, b_q} : M2{0.f, 0.f, 0.f, 0.f};
    const M2 dia = {fmaf(-a_d, P0, 1.f), fmaf(-a_d, Q0, a_g), -fmaf(b_g, P0, b_d * P1),
                    1.f - fmaf(b_g, Q0, b_d * Q1)};
    const M2 sup = {-a_d * R0, -a_d * S0, -fmaf(b_g, R0, b_d * R1), -fmaf(b_g, S0, b_d * S1)};
    const float2 rhs = {fmaf(-a_d, Y0, a_y), b_y - fmaf(b_g, Y0, b_d * Y1)};
    bool ok = true;
    // normalised block row: Xl t_{k-d} + t_k + Xr t_{k+d} = z
    const M2 di = inv(dia, ok);
    M2 Xl = mul(di, sub), Xr = mul(di, sup);
    float2 z = mul(di, rhs);
#pragma unroll
    for (int d = 1; d < P; d *= 2) {
      // lanes without a partner at k - d (k + d) have Xl (Xr) = 0 exactly, so
      // the values a shuffle returns for them drop out
      const M2 Xlm = shfl_up(Xl, d, P), Xrm = shfl_up(Xr, d, P);
      const float2 zm = {__shfl_up_sync(0xffffffffu, z.x, d, P), __shfl_up_sync(0xffffffffu, z.y, d, P)};
      const M2 Xlp = shfl_down(Xl, d, P), Xrp = shfl_down(Xr, d, P);
      const float2 zp = {__shfl_down_sync(0xffffffffu, z.x, d, P), __shfl_down_sync(0xffffffffu, z.y, d, P)};
      // substitute t_{k-d} and t_{k+d} from their rows:
      //   (I - Xl Xrm - Xr Xlp) t_k - Xl Xlm t_{k-2d} - Xr Xrp t_{k+2d} = z - Xl zm - Xr zp
      const M2 u1 = mul(Xl, Xrm), u2 = mul(Xr, Xlp);
      const M2 mm = {1.f - u1.a - u2.a, -u1.b - u2.b, -u1.c - u2.c, 1.f - u1.d - u2.d};
      const M2 mi = inv(mm, ok);
      const M2 nl = mul(Xl, Xlm), nr = mul(Xr, Xrp);
      const float2 a1 = mul(Xl, zm), a2 = mul(Xr, zp);
      const float2 zz = {z.x - a1.x - a2.x, z.y - a1.y - a2.y};
      const M2 l2 = mul(mi, nl), r2 = mul(mi, nr);
      Xl = {-l2.a, -l2.b, -l2.c, -l2.d};
      Xr = {-r2.a, -r2.b, -r2.c, -r2.d};
      z = mul(mi, zz);
    }
    if (!ok) atomicMin(&sBadR[q], min(N, (k + 1) * L));
    sT[0][k][q] = z.x;
    sT[1][k][q] = z.y;
  }
  __syncthreads();

  // ---- 4. every row from u = t_{c-1} and v = t_c
  const float u0 = c > 0 ? sT[0][c - 1][lane] : 0.f;
  const float u1 = c > 0 ? sT[1][c - 1][lane] : 0.f;
  const float v0 = sT[0][c][lane], v1 = sT[1][c][lane];
#pragma unroll
  for (int j = 0; j < L; ++j) {
    const int i = row0 + j;
    const float x = fmaf(-dl[j], v1, fmaf(-gm[j], v0, fmaf(-qq[j], u1, fmaf(-pp[j], u0, gg[j]))));
    if (act && i < N) X[(size_t)i * ld + sb] = x;
  }
  if (c == 0 && act && info) {
    // a failed local pivot also spoils the reduced system: report the pivot
    const int r = sBad[lane] != INT_MAX ? sBad[lane] : sBadR[lane];
    info[s] = r == INT_MAX ? 0 : r;
  }
}

template <int P>
cudaError_t launch(const void* a, const void* b, const void* c, const void* d, const void* e, void* X,
                   int N, int batch, int bs, int* info, cudaStream_t st) {
  const int grid = (batch + kSB - 1) / kSB;
  // TMA boxes of BR rows (even, <= 256) covering RS >= N rows
  const int BR = N <= 256 ? ((N + 1) & ~1) : 256;
  const int RS = (N + BR - 1) / BR * BR;
  PsMaps maps;
  const void* ptr[6] = {a, b, c, d, e, X};
  // a CTA's 16 systems must lie in one block of a block-interleaved array
  bool tma_ok = bs == 0 || bs % kSB == 0;
  for (int k = 0; k < 6 && tma_ok; ++k)
    tma_ok = bs ? tma::encode_3d_blocked(&maps.m[k], ptr[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sizeof(float),
                                         bs, N, batch / bs, kSB, (unsigned)BR)
                : tma::encode_2d(&maps.m[k], ptr[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sizeof(float), batch,
                                 N, kSB, (unsigned)BR);
  const size_t stage = tma_ok ? (size_t)6 * RS * kSB * sizeof(float)
                              : (size_t)6 * kL * kSB * P * sizeof(float);
  const size_t iface = (size_t)(kIface + 2) * P * (kSB + 1) * sizeof(float);
  const size_t smem = stage > iface ? stage : iface;
  auto kern = tma_ok ? k_persys_split<P, true> : k_persys_split<P, false>;
  const cudaError_t err = kernel_prepare((const void*)kern, smem, kSB * P, nullptr);
  if (err != cudaSuccess) return err;
  kern<<<grid, kSB * P, smem, st>>>(maps, static_cast<const float*>(a), static_cast<const float*>(b),
                                     static_cast<const float*>(c), static_cast<const float*>(d),
                                     static_cast<const float*>(e), static_cast<float*>(X), N, batch, bs,
                                     RS, BR, info);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

int persys_split_chunks(int N) {
  const int need = (N + kL - 1) / kL;
  int P = 2;
  while (P < need) P *= 2;
  return P <= 32 ? P : 0;
}

cudaError_t persys_split(const void* a, const void* b, const void* c, const void* d, const void* e, void* X,
                         int N, int batch, int bs, int* info, cudaStream_t st) {
  switch (persys_split_chunks(N)) {
    case 2: return launch<2>(a, b, c, d, e, X, N, batch, bs, info, st);
    case 4: return launch<4>(a, b, c, d, e, X, N, batch, bs, info, st);
    case 8: return launch<8>(a, b, c, d, e, X, N, batch, bs, info, st);
    case 16: return launch<16>(a, b, c, d, e, X, N, batch, bs, info, st);
    case 32: return launch<32>(a, b, c, d, e, X, N, batch, bs, info, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pent

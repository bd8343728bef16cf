// Fused time steps, one thread per system: explicit right-hand side + cyclic solve.
//
// Cahn–Hilliard (k_ch_thread_f64):
// "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs", eqs. (1a)
// and (2) with mobility D = 1, periodic on N points:
//   (I + gamma dt D4) C^{n+1} = C^n + dt D2[(C^n)^3 - C^n],  D2 = [1, -2, 1]/dx^2.
// The page builds the right-hand side with a separate stencil library before
// the solve.  Here the thread that solves system s computes its right-hand
// side on the fly inside the forward sweep: row i needs C_{i-1}, C_i, C_{i+1},
// all of which pass through the same thread, so the right-hand side never
// goes to memory.  The solve is the bordered cyclic sweep of pent_shared.cu.
//
// In-place safety: the forward sweep writes g_i over C_i only after C_{i+1}
// has been read, and rows N-2, N-1 (the border) are not overwritten until the
// end, so every C value is read before it is replaced.  C_{N-1} and C_0 are
// kept in registers for the periodic wrap.
//
// Crank–Nicolson (k_cn_thread_f64), eqs. (5)–(6) of the same page: with the
// plan's matrix A = I + sigma_x D4 (sigma_x = dt / (2 dx^4)) the explicit half
// I - sigma_x D4 equals 2I - A, so the right-hand side of row i is
//   2 C_i - (a_i C_{i-2} + b_i C_{i-1} + c_i C_i + d_i C_{i+1} + e_i C_{i+2})
// with the plan's own bands and periodic indices.  Any cyclic plan A = I + (dt/2) L
// gets its Crank–Nicolson step this way.  Row i reads C up to i+2 ahead and
// keeps C_{i-2}, C_{i-1} in registers; C_0, C_1, C_{N-2}, C_{N-1} are kept
// for the wrap.
#include "pent_internal.cuh"
#include "pent_native.cuh"

namespace pent {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
    k_ch_thread_f64(const double* __restrict__ coef, const double* __restrict__ tail,
                    double* __restrict__ X, int N, int batch, double k2) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  native_ch_column(coef, tail, X + s, N, (size_t)batch, k2);
}

__global__ void __launch_bounds__(kThreads)
    k_cn_thread_f64(const double* __restrict__ coef, const double* __restrict__ tail,
                    const double* __restrict__ bands, double* __restrict__ X, int N, int batch) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  native_cn_column(coef, tail, bands, X + s, N, (size_t)batch);
}

}  // namespace

cudaError_t ch_thread_f64(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  k_ch_thread_f64<<<grid, kThreads, 0, st>>>(p.coef64, p.tail64, X, p.N, batch, k2);
  note_launch();
  return cudaGetLastError();
}

cudaError_t cn_thread_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st) {
  const int grid = (batch + kThreads - 1) / kThreads;
  k_cn_thread_f64<<<grid, kThreads, 0, st>>>(p.coef64, p.tail64, p.bands, X, p.N, batch);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pent

// Internal declarations of libpent: plan layout, coefficient tables, launchers.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "pent.h"

namespace pent {

// Per-row coefficient tables of a factored shared matrix, stored as
// [kCoefCount][M] arrays (M = rows swept: N, or N-2 for a cyclic plan).
//   forward   g_i = r_i f_i - p_i g_{i-2} - q_i g_{i-1}
//             with r = 1/alpha, p = eps/alpha, q = beta/alpha
//   backward  y_i = g_i - gamma_i y_{i+1} - delta_i y_{i+2}
//   cyclic    acc_k += w_k,i g_i  (w_k = R^{-T} h_k, so sum_i w_k,i g_i = h_k^T E^{-1} f)
//             x_i = y_i - u0_i x_{N-2} - u1_i x_{N-1}  (u_k = E^{-1} G_k)
enum Coef : int { kR = 0, kP, kQ, kW0, kW1, kGam, kDel, kU0, kU1, kCoefCount };

// tail[0..3] = (B - H^T E^{-1} G)^{-1} row-major (cyclic plans only).
constexpr int kTailCount = 4;

}  // namespace pent

struct pent_plan_s {
  int N = 0, M = 0, batch = 0, cyclic = 0;
  pent_dtype dtype = PENT_F64;
  pent_variant variant = PENT_VARIANT_AUTO;
  int device = 0;
  double* coef64 = nullptr;  // [kCoefCount][M] fp64
  double* tail64 = nullptr;  // [4]
  float* coef32 = nullptr;   // [kCoefCount][M] fp32 (fp32 plans)
  float* tail32 = nullptr;
  float2* coefdf = nullptr;  // [kCoefCount][M] (hi, lo) double-float pairs
  float2* taildf = nullptr;
  void* arena = nullptr;     // single allocation backing all of the above
  // twisted double-float variant (pent_factor_twisted.cu / pent_shared_df.cu)
  int m = 0;                 // meeting row: top rows 0..m-1, bottom rows m..M-1
  int twist_ok = 0;          // tables valid and the 4x4 meeting system nonsingular
  float4* twtab = nullptr;   // [M][kTwK]
  double* twist = nullptr;   // [kTwistCount]
  int num_sms = 0;           // SMs of the plan's device (persistent grid size)
  int df_spb = 128;          // systems per CTA of the double-float kernels
  int df_ctas = 0;           // CTAs of the double-float kernels (0: one per SM)
};

namespace pent {

// launch bookkeeping (host)
void note_launch();

// factor.cu
cudaError_t factor_shared(const double* d_bands, int N, int cyclic, double* coef64, double* tail64,
                          double* d_work, int* d_status, cudaStream_t st);
cudaError_t pack_coefficients(const double* coef64, const double* tail64, int n_coef, float* coef32,
                              float* tail32, float2* coefdf, float2* taildf, cudaStream_t st);

// shared.cu
cudaError_t shared_thread_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st);
cudaError_t shared_thread_f32(const pent_plan_s& p, float* X, int batch, cudaStream_t st);
cudaError_t shared_thread_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st);
cudaError_t shared_split_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st);
size_t shared_df_smem_bytes(int M);

// persys.cu
cudaError_t persys_thread(const void* a, const void* b, const void* c, const void* d, const void* e,
                          void* X, int N, int batch, pent_dtype dt, void* work, int* info,
                          cudaStream_t st);
size_t persys_work_bytes(int N, int batch, pent_dtype dt);

// ch.cu
cudaError_t ch_thread_f64(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st);
cudaError_t ch_thread_df(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st);

}  // namespace pent

namespace pent {

// Twisted (two-sided) factorisation tables for the double-float kernels.
// The M-row block is swept by two threads per system: "top" runs the LR
// recurrences over rows 0..m-1, "bottom" runs the same recurrences on the
// reversed block over rows M-1..m; a 4x4 system couples them at the middle.
// Per table row, kTwK float4 of (hi, lo) pairs:
//   k0 = {r, P}    inward   g_j = r_j f_j + P_j g_{j-2} + Q_j g_{j-1}
//   k1 = {Q, C}    outward  y_j = g_j + C_j y_{j+1} + D_j y_{j+2}
//   k2 = {D, q0}   cyclic:  acc_k += q_k f_j  (q_k = E^{-T} h_k)
//   k3 = {q1, u0}           x = y - u0 x_t0 - u1 x_t1  (u_k = E^{-1} G_k)
//   k4 = {u1, 0}
// Table rows 0..m-1 are the top direction, rows m..M-1 the bottom direction
// (local row j at table row m + j, global row M-1-j).
constexpr int kTwK = 5;
// twist[0..15] = T^{-1} (row-major, unknowns x_{m-2}, x_{m-1}, x_m, x_{m+1});
// twist[16..19] = S^{-1} of the border (cyclic plans).
constexpr int kTwistCount = 20;

cudaError_t factor_twisted(const double* d_bands, int N, int cyclic, int m, float4* tab,
                           double* twist, double* d_work, int* d_status, cudaStream_t st);

}  // namespace pent

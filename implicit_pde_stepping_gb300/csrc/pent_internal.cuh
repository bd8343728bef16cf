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
  double* bands = nullptr;   // [5][N] the matrix as factored (a, b, c, d, e)
  void* arena = nullptr;     // single allocation backing all of the above
  // twisted double-float variant (pent_factor_twisted.cu / pent_twisted_df.cu)
  int m = 0;                 // meeting row: top rows 0..m-1, bottom rows m..M-1
  int twist_ok = 0;          // tables valid and the 4x4 meeting system nonsingular
  int twist_eligible = 0;    // fp64 plan whose block suits the twisted kernel
  int twist_built = 0;       // tables made (on first selection of the variant)
  double* work_area = nullptr;   // plan-time scratch in the arena
  int* status_area = nullptr;
  float4* twtab = nullptr;   // [M][kTwK]
  double* twist = nullptr;   // [kTwistCount]
  int num_sms = 0;           // SMs of the plan's device (persistent grid size)
  int df_spb = 256;          // systems per CTA of the double-float kernels
  int df_spt = 2;            // systems per thread (2 needs an even batch)
  int df_ku = 4;             // rows per prefetch block
  int df_ctas = 0;           // CTAs of the double-float kernels (0: two per SM)
  int steps_sb = 0;          // systems per CTA of the multi-step kernel (0: chosen by shape)
  int df_async = 6;          // cp.async ring depth of the twisted kernel (0: register ring)
  int steps_on = 1;          // multi-step kernel for nsteps >= 2 where supported
  // as found when the plan was built (pent_set_option switches back to them)
  int sp_T0 = 0, reach0 = 0, cheap_k0 = 0, cheap_m0 = 1 << 20, dup_lo0 = 0, dup_hi0 = 0;
  // partitioned double-float variant (pent_factor_split.cu / pent_split_df.cu)
  int split_ok = 0;          // tables valid
  int sp_L = 0, sp_P = 0;    // chunk length, chunks per system (Mpad = sp_L * sp_P)
  int sp_T = 0;              // chunk couplings kept by the parallel scan (0: exact serial scan)
  int split_big = 0;         // tables valid for the two-kernel form (systems too long for one CTA)
  double* spsum = nullptr;   // two-kernel form: per system and chunk summaries, grown on use
  // chunks dup_lo < c <= dup_hi have row and chunk tables bitwise equal to those of
  // chunk dup_lo (a matrix with constant bands, far from its ends): the two-kernel
  // form reads chunk dup_lo's tables for them, which stay in cache
  int dup_lo = 0, dup_hi = 0;
  // in the 8-row groups g < cheap_k of every chunk the responses K1, K2 to the
  // chunk's outgoing state, in the groups g >= cheap_m the responses M1, M2 to its
  // incoming state, are below 2^-24 in every chunk; the multi-step kernel then adds
  // their correction terms to the low word alone (one FMA instead of a double-float
  // multiply-add, at most about 3 * 2^-48 of the state per term)
  int cheap_k = 0, cheap_m = 1 << 20;
  size_t spsum_bytes = 0;
  // fixed-grid partitioned kernel (pent_fg.cu): valid for this plan, grid bias,
  // correction-term groups (see fg_prepare), bound on the intermediate values
  int fg_ok = 0;
  int big_fg = 0;             // the long-system kernels may use the grid (fg_bias)
  int fg_use = 1;            // test option: 0 keeps the TwoSum double-float kernel
  float fg_bias = 0.f;
  int fg_gm_full = 0, fg_gm_none = 0, fg_gk_none = 0, fg_gk_full = 0;
  int fg_dup_lo = 0, fg_dup_hi = 0;   // chunks dup_lo < c <= dup_hi share chunk dup_lo's row tables
  int* kern_err = nullptr;   // device word: 1 once a kernel gave up waiting for a tile copy
  unsigned* sched = nullptr; // device words {next block, CTAs done} of the persistent solve's
                             // block queue; zero between launches (the last CTA resets them)
  double fg_bound = 0.0;
  float4* sptab = nullptr;   // [Mpad][kSpK]
  double* spchunk = nullptr; // [sp_P][kSpChunk]
  float2* spchunk_df = nullptr;   // the same as double-float pairs (the scans on the FP32 pipe)
  double* spextra = nullptr; // [kSpExtra]
  // host-buffer pipeline (pent_host.cu), created on first use
  static constexpr int kHostRing = 3;
  cudaStream_t hs[3] = {nullptr, nullptr, nullptr};   // copy in, solve, copy out
  cudaEvent_t hev_in[kHostRing] = {}, hev_solved[kHostRing] = {}, hev_out[kHostRing] = {};
  cudaEvent_t hev_fork = nullptr;
  void* hbuf = nullptr;       // kHostRing staging buffers of hbuf_bytes each
  size_t hbuf_bytes = 0;
};

namespace pent {

// launch bookkeeping (host)
void note_launch();
// Raise kernel fn's dynamic shared-memory limit to smem bytes on the current
// device and, if per_sm is not null, report how many CTAs of `threads` threads
// fit on one SM.  Both are cached per kernel, device and size, so repeated
// launches make no attribute or occupancy call (each costs microseconds of host
// time, which a short kernel's stream would otherwise wait through).
cudaError_t kernel_prepare(const void* fn, size_t smem, int threads, int* per_sm);

// factor.cu
cudaError_t factor_shared(const double* d_bands, int N, int cyclic, double* coef64, double* tail64,
                          double* d_work, int* d_status, cudaStream_t st);
cudaError_t pack_coefficients(const double* coef64, const double* tail64, int n_coef, float* coef32,
                              float* tail32, float2* coefdf, float2* taildf, cudaStream_t st);

// shared.cu
cudaError_t shared_thread_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st);
cudaError_t shared_thread_f32(const pent_plan_s& p, float* X, int batch, cudaStream_t st);
cudaError_t shared_twisted_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st);

// persys.cu
// bs = 0: interleaved [N][batch]; bs > 0: block-interleaved, blocks of bs systems
cudaError_t persys_thread(const void* a, const void* b, const void* c, const void* d, const void* e,
                          void* X, int N, int batch, int bs, pent_dtype dt, void* work, int* info,
                          cudaStream_t st);
size_t persys_work_bytes(int N, int batch, pent_dtype dt);
// fp64 matrices computed in double-float (same scratch size as persys_thread)
cudaError_t persys_thread_df(const void* a, const void* b, const void* c, const void* d, const void* e,
                             void* X, int N, int batch, int bs, void* work, int* info, cudaStream_t st);
// persys_split.cu: partitioned fp32 kernel (chunks of 16 rows, TMA tiles)
int persys_split_chunks(int N);   // chunks per system for N rows, 0 if N > 512
cudaError_t persys_split(const void* a, const void* b, const void* c, const void* d, const void* e, void* X,
                         int N, int batch, int bs, int* info, cudaStream_t st);

// tri.cu: per-system tridiagonal solves (Thomas algorithm; partitioned fp32 kernel)
int tri_split_chunks(int N);   // chunks of the partitioned kernel for N rows, 0 if too large
size_t tri_work_bytes(int N, int batch, pent_dtype dt);
// bs = 0: interleaved [N][batch]; bs > 0: block-interleaved, blocks of bs systems
cudaError_t tri_solve_batch(const void* a, const void* b, const void* c, void* X, int N, int batch, int bs,
                            pent_dtype dt, bool split, void* work, int* info, cudaStream_t st);
// fp64 systems in double-float, one thread per system (same scratch size)
cudaError_t tri_solve_batch_df(const void* a, const void* b, const void* c, void* X, int N, int batch, int bs,
                               void* work, int* info, cudaStream_t st);

// host.cu: shared-matrix solve of host arrays, transfers overlapped with the solves
void host_pipeline_release(pent_plan_s& p);
cudaError_t solve_host(pent_plan_s& p, const void* in, void* out, int batch, int chunks, cudaStream_t st,
                       cudaError_t (*solve)(pent_plan_s&, void*, int, cudaStream_t));
// api.cu: the plan's solve kernel, in place on a device array (leading dimension batch)
cudaError_t solve_device(pent_plan_s& p, void* rhs, int batch, cudaStream_t st);

// ch.cu: fused explicit right-hand side + cyclic solve, one thread per system
cudaError_t ch_thread_f64(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st);
cudaError_t cn_thread_f64(const pent_plan_s& p, double* X, int batch, cudaStream_t st);

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
// twist[16..19] = S^{-1} of the border (cyclic plans); twist[20] = border reach W
// (cyclic): only local rows j < W of either direction carry a q or u entry of
// magnitude >= 2^-60, so the others skip the border terms; [21..23] unused (the
// kernels keep this table in shared memory, and a size that is a multiple of 32
// bytes keeps the dynamic shared memory after it aligned: 21 entries cost the
// headline solve 12%).
constexpr int kTwistCount = 24;

cudaError_t factor_twisted(const double* d_bands, int N, int cyclic, int m, float4* tab,
                           double* twist, double* d_work, int* d_status, cudaStream_t st);

}  // namespace pent

namespace pent {

// Partitioned ("split") double-float kernel tables (pent_factor_split.cu).
// The M-row block is padded to Mpad = P * L rows (padding rows are decoupled
// identity rows) and cut into P chunks of L rows.  Per padded row, kSpK float4
// of (hi, lo) pairs:
//   k0 = {r, P}   k1 = {Q, U0}   k2 = {C, D}   k3 = {M1, M2}   k4 = {K1, K2}   k5 = {U1, 0}
// forward  g_j = r f + P g_{j-2} + Q g_{j-1}; backward y_j = g_j + C y_{j+1} + D y_{j+2};
// H1/H2 = forward responses of a chunk to its incoming state (g_{a-2}, g_{a-1}),
// M1/M2 = their local back substitution, K1/K2 = backward responses to the
// outgoing state (x_b, x_{b+1}); U0/U1 = E^{-1} G (cyclic).
constexpr int kSpK = 6;
// Per chunk c, kSpChunk doubles, each 2x2 row-major:
//   [0]  Phi_c  (H at the chunk's last two rows: s_{c+1} = e_c + Phi_c s_c)
//   [4]  Mst_c  (M at its first two rows)    [8] Kst_c (K at its first two rows)
//   [12 + 4(k-2)]  A_{c,k} = Phi_{c-1} ... Phi_{c-k+1},  k = 2..kSpTmax
//   [24 + 4(k-1)]  B_{c,k} = Kst_{c+1} ... Kst_{c+k},    k = 1..kSpTmax-1
// so that s_c = sum_{k=1..T} A_{c,k} e_{c-k} (A_{c,1} = I) and
// t_c = sum_{k=0..T-1} B_{c,k} w_{c+1+k} (B_{c,0} = I), w_c = x'_start(c) + Mst_c s_c.
constexpr int kSpTmax = 4;
constexpr int kSpMaxChunks = 64;   // chunks per system the split kernel supports
constexpr int kSpChunk = 36;
// Extras: [0..3] S^{-1} (cyclic); [4..6] h0 at rows M-2, M-1, 0; [7..9] h1 at rows
// M-1, 0, 1; [10..13] M1,M2 at rows M-2 then M-1; [14..17] K1,K2 at rows M-2 then
// M-1; [18] T, the number of chunk couplings kept (0: exact serial scan); [19] the
// border reach R (cyclic): only chunks c < R or c > (M-1)/L - R carry a
// non-negligible E^{-1} G and apply the x_t correction.
constexpr int kSpExtra = 20;

cudaError_t factor_split(const double* d_bands, int N, int cyclic, int L, int Mpad, float4* rowtab,
                         double* chunktab, double* extra, double* d_work, int* d_status,
                         cudaStream_t st);
cudaError_t shared_split_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st);
// pent_split_big.cu: the same solve for systems too long for one CTA (two kernels)
cudaError_t shared_split_big(pent_plan_s& p, double* X, int batch, cudaStream_t st);
// plan time: the double-float copy of the chunk tables
cudaError_t split_big_prepare(pent_plan_s& p, cudaStream_t st);
size_t split_smem_bytes(int L, int P, int SB, int cyclic);
cudaError_t ch_split_df(const pent_plan_s& p, double* X, int batch, double k2, cudaStream_t st);
cudaError_t cn_split_df(const pent_plan_s& p, double* X, int batch, cudaStream_t st);

// pent_fg.cu: the partitioned solve in fixed-grid double-float (non-cyclic
// plans with L = 32 chunks and a truncated chunk scan); fg_prepare decides at
// plan time whether it applies and sets its grid
cudaError_t fg_prepare(pent_plan_s& p);
cudaError_t shared_fg(const pent_plan_s& p, double* X, int batch, cudaStream_t st);

// pent_steps_df.cu: nsteps of a periodic scheme in one launch, state in registers.
// kind 0 = hyperdiffusion, 1 = Cahn–Hilliard (k2 = dt/dx^2), 2 = Crank–Nicolson.
constexpr size_t kStepsSmemMax = 227 * 1024;
bool steps_supported(const pent_plan_s& p, int kind);
cudaError_t steps_df(const pent_plan_s& p, double* X, int batch, int nsteps, int kind, double k2,
                     cudaStream_t st);

}  // namespace pent

/*
 * Reference oracle for batched pentadiagonal solves — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct CPU code in fp64.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant with the CUDA library: the two are independent
 * implementations of the same mathematics, and parity between them is what the
 * GPU tests check.
 *
 * Source followed throughout: "cuPentBatch – A batched pentadiagonal solver
 * for NVIDIA GPUs" (Gloster et al., arXiv 1807.07382).
 *   - pentadiagonal LR factorisation, factorisation steps 1–14;
 *   - forward substitution L g = f, steps 1–3;
 *   - back substitution R x = g, steps 1–3;
 *   - periodic (cyclic) matrix (7c) solved by Navon's bordering, eqs. (8)–(12);
 *   - hyperdiffusion / Cahn–Hilliard semi-implicit stepping, eqs. (1)–(2), (4);
 *   - Crank–Nicolson hyperdiffusion, eqs. (5)–(6), sigma_x = dt / (2 dx^4).
 * And, from "Simulating the behavior of the human brain on GPUs" (Valero-Lara
 * et al.), section 4.1 "Tridiagonal linear systems":
 *   - the Thomas algorithm: forward elimination of the lower diagonal
 *     (c'_i, y'_i), then backward substitution u_i = y'_i - c'_i u_{i+1}.
 *     Its tridiagonal rows: a_i below the diagonal (column i-1), b_i on it,
 *     c_i above it (column i+1); a_0 and c_{N-1} do not exist.
 *
 * Conventions (0-based; the page is 1-based).  Row i of the matrix holds
 *   a[i] at column i-2, b[i] at i-1, c[i] at i, d[i] at i+1, e[i] at i+2.
 * This naming is the one the factorisation steps use (alpha_1 = c_1,
 * beta_2 = b_2, gamma_1 = d_1/alpha_1, delta_1 = e_1/alpha_1, eps_i = a_i).
 * For a non-cyclic matrix, entries whose column falls outside 0..N-1 are
 * ignored (treated as zero).  For a cyclic matrix the column wraps mod N.
 *
 * Loop form.  The page writes the first two and last two rows of each sweep
 * out by hand and loops over the interior.  Here one loop runs over every row,
 * with every quantity of an out-of-range index taken as zero.  Because
 * x - 0*y == x exactly in IEEE arithmetic, this gives bit-for-bit the page's
 * unrolled steps for N >= 4 and also defines N = 1..3.
 *
 * Systems in a batch are stored one per row ("row-major, one system per
 * row"), the layout of the page's serial C validation code.  The batch loops
 * are parallelised over systems with OpenMP when it is available, as in the
 * page's OpenMP comparison (same serial code, batch loop parallel).
 *
 * Return codes: 0 ok, 1 invalid argument, 2 zero pivot (alpha == 0 or a
 * singular 2x2 border block), 3 out of memory.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_OK = 0, OR_EINVAL = 1, OR_ZERO_PIVOT = 2, OR_ENOMEM = 3 };

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Band value of row i for the non-cyclic matrix: out-of-range columns are 0. */
static double band_nc(const double* v, int i, int off, int N) {
  int col = i + off;
  if (col < 0 || col >= N) return 0.0;
  return v[i];
}

/*
 * Pentadiagonal LR factorisation (factorisation steps 1–14).
 *   beta_i  = b_i - a_i gamma_{i-2}
 *   alpha_i = c_i - a_i delta_{i-2} - beta_i gamma_{i-1}
 *   gamma_i = (d_i - beta_i delta_{i-1}) / alpha_i
 *   delta_i = e_i / alpha_i
 *   eps_i   = a_i
 * Out-of-range bands are zero (non-cyclic matrix).
 */
int oracle_pent_factor(int N, const double* a, const double* b, const double* c, const double* d,
                       const double* e, double* alpha, double* beta, double* gamma, double* delta,
                       double* eps) {
  if (N < 1) return OR_EINVAL;
  for (int i = 0; i < N; ++i) {
    double ai = band_nc(a, i, -2, N), bi = band_nc(b, i, -1, N), ci = c[i];
    double di = band_nc(d, i, +1, N), ei = band_nc(e, i, +2, N);
    double gm2 = (i >= 2) ? gamma[i - 2] : 0.0, dm2 = (i >= 2) ? delta[i - 2] : 0.0;
    double gm1 = (i >= 1) ? gamma[i - 1] : 0.0, dm1 = (i >= 1) ? delta[i - 1] : 0.0;
    beta[i] = bi - ai * gm2;
    alpha[i] = ci - ai * dm2 - beta[i] * gm1;
    if (alpha[i] == 0.0 || !isfinite(alpha[i])) return OR_ZERO_PIVOT;
    gamma[i] = (di - beta[i] * dm1) / alpha[i];
    delta[i] = ei / alpha[i];
    eps[i] = ai;
  }
  return OR_OK;
}

/* Forward substitution L g = f:  g_i = (f_i - eps_i g_{i-2} - beta_i g_{i-1}) / alpha_i. */
void oracle_pent_forward(int N, const double* alpha, const double* beta, const double* eps,
                         const double* f, double* g) {
  for (int i = 0; i < N; ++i) {
    double gm2 = (i >= 2) ? g[i - 2] : 0.0, gm1 = (i >= 1) ? g[i - 1] : 0.0;
    g[i] = (f[i] - eps[i] * gm2 - beta[i] * gm1) / alpha[i];
  }
}

/* Back substitution R x = g:  x_i = g_i - gamma_i x_{i+1} - delta_i x_{i+2}. */
void oracle_pent_backward(int N, const double* gamma, const double* delta, const double* g,
                          double* x) {
  for (int i = N - 1; i >= 0; --i) {
    double xp1 = (i + 1 < N) ? x[i + 1] : 0.0, xp2 = (i + 2 < N) ? x[i + 2] : 0.0;
    x[i] = g[i] - gamma[i] * xp1 - delta[i] * xp2;
  }
}

/* Factor + forward + backward for one non-cyclic system (x may alias f). */
int oracle_pent_solve(int N, const double* a, const double* b, const double* c, const double* d,
                      const double* e, const double* f, double* x) {
  if (N < 1) return OR_EINVAL;
  double* w = (double*)malloc(sizeof(double) * 6 * (size_t)N);
  if (!w) return OR_ENOMEM;
  double *alpha = w, *beta = w + N, *gamma = w + 2 * N, *delta = w + 3 * N, *eps = w + 4 * N,
         *g = w + 5 * N;
  int rc = oracle_pent_factor(N, a, b, c, d, e, alpha, beta, gamma, delta, eps);
  if (rc == OR_OK) {
    oracle_pent_forward(N, alpha, beta, eps, f, g);
    oracle_pent_backward(N, gamma, delta, g, x);
  }
  free(w);
  return rc;
}

/*
 * Cyclic pentadiagonal solve by Navon's bordering (eqs. (8)–(12)).
 * A is split as [[E, G], [H^T, B]] with E the leading (N-2)x(N-2) block,
 * G the last two columns of the first N-2 rows, H^T the first N-2 columns of
 * the last two rows and B the trailing 2x2 block.  Each piece is assembled
 * entry by entry from the wrapped column index.  Then
 *   Y_f = E^{-1} f_hat,  Y_G = E^{-1} G                (pentadiagonal solves of E)
 *   S   = B - H^T Y_G                                  (2x2)
 *   x_t = S^{-1} (f_t - H^T Y_f)                       (eq. (12), Cramer's rule)
 *   x_hat = Y_f - Y_G x_t                              (eq. (11))
 * Requires N >= 5 so that the five columns of a row are distinct.
 */
int oracle_cyclic_solve(int N, const double* a, const double* b, const double* c, const double* d,
                        const double* e, const double* f, double* x) {
  if (N < 5) return OR_EINVAL;
  const int M = N - 2;
  const double* band[5] = {a, b, c, d, e};
  double* w = (double*)calloc((size_t)M * 11, sizeof(double));
  if (!w) return OR_ENOMEM;
  double *Ea = w, *Eb = w + M, *Ec = w + 2 * M, *Ed = w + 3 * M, *Ee = w + 4 * M;
  double *G0 = w + 5 * M, *G1 = w + 6 * M, *H0 = w + 7 * M, *H1 = w + 8 * M;
  double *Yf = w + 9 * M, *Y0 = w + 10 * M;
  double* Eband[5] = {Ea, Eb, Ec, Ed, Ee};
  double Bm[2][2] = {{0.0, 0.0}, {0.0, 0.0}};
  double* Y1 = (double*)malloc(sizeof(double) * (size_t)M);
  if (!Y1) { free(w); return OR_ENOMEM; }
  /* Assemble E, G, H^T, B from the wrapped columns. */
  for (int i = 0; i < N; ++i) {
    for (int k = 0; k < 5; ++k) {
      int col = ((i + k - 2) % N + N) % N;
      double v = band[k][i];
      if (i < M && col < M) {
        /* inside E: col - i is k - 2 (no wrap can land inside E for N >= 5) */
        Eband[k][i] += v;
      } else if (i < M) {
        if (col == M) G0[i] += v; else G1[i] += v;
      } else if (col < M) {
        if (i == M) H0[col] += v; else H1[col] += v;
      } else {
        Bm[i - M][col - M] += v;
      }
    }
  }
  int rc = oracle_pent_solve(M, Ea, Eb, Ec, Ed, Ee, f, Yf);
  if (rc == OR_OK) rc = oracle_pent_solve(M, Ea, Eb, Ec, Ed, Ee, G0, Y0);
  if (rc == OR_OK) rc = oracle_pent_solve(M, Ea, Eb, Ec, Ed, Ee, G1, Y1);
  if (rc == OR_OK) {
    double S00 = Bm[0][0], S01 = Bm[0][1], S10 = Bm[1][0], S11 = Bm[1][1];
    double r0 = f[M], r1 = f[M + 1];
    for (int j = 0; j < M; ++j) {
      S00 -= H0[j] * Y0[j];
      S01 -= H0[j] * Y1[j];
      S10 -= H1[j] * Y0[j];
      S11 -= H1[j] * Y1[j];
      r0 -= H0[j] * Yf[j];
      r1 -= H1[j] * Yf[j];
    }
    double det = S00 * S11 - S01 * S10;
    if (det == 0.0 || !isfinite(det)) {
      rc = OR_ZERO_PIVOT;
    } else {
      double xt0 = (r0 * S11 - S01 * r1) / det;
      double xt1 = (S00 * r1 - S10 * r0) / det;
      for (int j = 0; j < M; ++j) x[j] = Yf[j] - Y0[j] * xt0 - Y1[j] * xt1;
      x[M] = xt0;
      x[M + 1] = xt1;
    }
  }
  free(w); free(Y1);
  return rc;
}

/* Bands of I + sigma * D4 with D4 the centred [1, -4, 6, -4, 1] stencil. */
static void hyper_bands(int N, double sigma, double* a, double* b, double* c, double* d, double* e) {
  for (int i = 0; i < N; ++i) {
    a[i] = sigma; b[i] = -4.0 * sigma; c[i] = 1.0 + 6.0 * sigma; d[i] = -4.0 * sigma; e[i] = sigma;
  }
}

/* nsteps of C <- (I + sigma D4)^{-1} C, periodic (cyclic matrix (7c)). */
int oracle_hyperdiffusion_steps(int N, double sigma, int nsteps, double* C) {
  if (N < 5 || nsteps < 0) return OR_EINVAL;
  double* w = (double*)malloc(sizeof(double) * 6 * (size_t)N);
  if (!w) return OR_ENOMEM;
  double *a = w, *b = w + N, *c = w + 2 * N, *d = w + 3 * N, *e = w + 4 * N, *x = w + 5 * N;
  hyper_bands(N, sigma, a, b, c, d, e);
  int rc = OR_OK;
  for (int n = 0; n < nsteps && rc == OR_OK; ++n) {
    rc = oracle_cyclic_solve(N, a, b, c, d, e, C, x);
    if (rc == OR_OK) memcpy(C, x, sizeof(double) * (size_t)N);
  }
  free(w);
  return rc;
}

/*
 * nsteps of the semi-implicit Cahn–Hilliard scheme (eq. (2), mobility D = 1),
 * periodic:  (I + sigma D4) C^{n+1} = C^n + (dt/dx^2) D2[(C^n)^3 - C^n],
 * D2 the centred [1, -2, 1] stencil, sigma = gamma dt / dx^4.
 */
int oracle_ch_steps(int N, double sigma, double dt_over_dx2, int nsteps, double* C) {
  if (N < 5 || nsteps < 0) return OR_EINVAL;
  double* w = (double*)malloc(sizeof(double) * 8 * (size_t)N);
  if (!w) return OR_ENOMEM;
  double *a = w, *b = w + N, *c = w + 2 * N, *d = w + 3 * N, *e = w + 4 * N, *x = w + 5 * N;
  double *u = w + 6 * N, *rhs = w + 7 * N;
  hyper_bands(N, sigma, a, b, c, d, e);
  int rc = OR_OK;
  for (int n = 0; n < nsteps && rc == OR_OK; ++n) {
    for (int i = 0; i < N; ++i) u[i] = C[i] * C[i] * C[i] - C[i];
    for (int i = 0; i < N; ++i) {
      int im = (i + N - 1) % N, ip = (i + 1) % N;
      rhs[i] = C[i] + dt_over_dx2 * (u[im] - 2.0 * u[i] + u[ip]);
    }
    rc = oracle_cyclic_solve(N, a, b, c, d, e, rhs, x);
    if (rc == OR_OK) memcpy(C, x, sizeof(double) * (size_t)N);
  }
  free(w);
  return rc;
}

/*
 * nsteps of the Crank–Nicolson scheme for hyperdiffusion, periodic
 * (eqs. (5)–(6), sigma_x = dt / (2 dx^4)):
 *   (I + sigma_x D4) C^{n+1} = (I - sigma_x D4) C^n.
 * The right-hand side is the explicit stencil applied to C^n, indices mod N.
 */
int oracle_cn_steps(int N, double sigma_x, int nsteps, double* C) {
  if (N < 5 || nsteps < 0) return OR_EINVAL;
  double* w = (double*)malloc(sizeof(double) * 7 * (size_t)N);
  if (!w) return OR_ENOMEM;
  double *a = w, *b = w + N, *c = w + 2 * N, *d = w + 3 * N, *e = w + 4 * N, *x = w + 5 * N;
  double* rhs = w + 6 * N;
  hyper_bands(N, sigma_x, a, b, c, d, e);
  int rc = OR_OK;
  for (int n = 0; n < nsteps && rc == OR_OK; ++n) {
    for (int i = 0; i < N; ++i) {
      int im2 = (i + N - 2) % N, im1 = (i + N - 1) % N, ip1 = (i + 1) % N, ip2 = (i + 2) % N;
      double d4 = C[im2] - 4.0 * C[im1] + 6.0 * C[i] - 4.0 * C[ip1] + C[ip2];
      rhs[i] = C[i] - sigma_x * d4;
    }
    rc = oracle_cyclic_solve(N, a, b, c, d, e, rhs, x);
    if (rc == OR_OK) memcpy(C, x, sizeof(double) * (size_t)N);
  }
  free(w);
  return rc;
}

/*
 * Thomas algorithm (section 4.1 of the tridiagonal page), one system:
 *   c'_0 = c_0 / b_0,   c'_i = c_i / (b_i - c'_{i-1} a_i),
 *   y'_0 = y_0 / b_0,   y'_i = (y_i - y'_{i-1} a_i) / (b_i - c'_{i-1} a_i),
 *   u_{N-1} = y'_{N-1}, u_i = y'_i - c'_i u_{i+1}.
 * a[0] and c[N-1] are ignored.  A zero denominator is a zero pivot.
 */
int oracle_tri_solve(int N, const double* a, const double* b, const double* c, const double* y,
                     double* u) {
  if (N < 1) return OR_EINVAL;
  double* cp = (double*)malloc(sizeof(double) * 2 * (size_t)N);
  if (!cp) return OR_ENOMEM;
  double* yp = cp + N;
  for (int i = 0; i < N; ++i) {
    const double ai = i > 0 ? a[i] : 0.0;
    const double ci = i + 1 < N ? c[i] : 0.0;
    const double cprev = i > 0 ? cp[i - 1] : 0.0;
    const double yprev = i > 0 ? yp[i - 1] : 0.0;
    const double den = b[i] - cprev * ai;
    if (den == 0.0 || !isfinite(den)) {
      free(cp);
      return OR_ZERO_PIVOT;
    }
    cp[i] = ci / den;
    yp[i] = (y[i] - yprev * ai) / den;
  }
  u[N - 1] = yp[N - 1];
  for (int i = N - 2; i >= 0; --i) u[i] = yp[i] - cp[i] * u[i + 1];
  free(cp);
  return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Batched drivers.  X and F are [batch][N] (one system per row); X may alias F.
 * Each returns the first nonzero per-system code, or 0.
 * ------------------------------------------------------------------------- */

/* Shared bands [5][N] (a, b, c, d, e), non-cyclic or cyclic.  For the
 * non-cyclic case the factorisation is done once and reused for every system
 * (factor once, solve many); the cyclic case applies the bordering solve to
 * each system. */
int oracle_batch_shared(int N, int batch, const double* bands, int cyclic, const double* F,
                        double* X) {
  if (N < 1 || batch < 0 || (cyclic && N < 5)) return OR_EINVAL;
  const double *a = bands, *b = bands + N, *c = bands + 2 * (size_t)N, *d = bands + 3 * (size_t)N,
               *e = bands + 4 * (size_t)N;
  int rc = OR_OK;
  if (!cyclic) {
    double* w = (double*)malloc(sizeof(double) * 5 * (size_t)N);
    if (!w) return OR_ENOMEM;
    double *alpha = w, *beta = w + N, *gamma = w + 2 * N, *delta = w + 3 * N, *eps = w + 4 * N;
    rc = oracle_pent_factor(N, a, b, c, d, e, alpha, beta, gamma, delta, eps);
    if (rc == OR_OK) {
#pragma omp parallel
      {
        double* g = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(static)
        for (long s = 0; s < batch; ++s) {
          if (!g) continue;
          oracle_pent_forward(N, alpha, beta, eps, F + s * (size_t)N, g);
          oracle_pent_backward(N, gamma, delta, g, X + s * (size_t)N);
        }
        if (!g) {
#pragma omp atomic write
          rc = OR_ENOMEM;
        }
        free(g);
      }
    }
    free(w);
    return rc;
  }
#pragma omp parallel for schedule(static)
  for (long s = 0; s < batch; ++s) {
    int r = oracle_cyclic_solve(N, a, b, c, d, e, F + s * (size_t)N, X + s * (size_t)N);
    if (r != OR_OK) {
#pragma omp critical
      if (rc == OR_OK) rc = r;
    }
  }
  return rc;
}

/* Per-system bands, each array [batch][N]; full factor + solve per system. */
int oracle_batch_persys(int N, int batch, const double* A, const double* B, const double* Cd,
                        const double* D, const double* E, const double* F, double* X) {
  if (N < 1 || batch < 0) return OR_EINVAL;
  int rc = OR_OK;
#pragma omp parallel for schedule(static)
  for (long s = 0; s < batch; ++s) {
    size_t o = s * (size_t)N;
    int r = oracle_pent_solve(N, A + o, B + o, Cd + o, D + o, E + o, F + o, X + o);
    if (r != OR_OK) {
#pragma omp critical
      if (rc == OR_OK) rc = r;
    }
  }
  return rc;
}

int oracle_batch_hyperdiffusion(int N, int batch, double sigma, int nsteps, double* C) {
  if (N < 5 || batch < 0) return OR_EINVAL;
  int rc = OR_OK;
#pragma omp parallel for schedule(static)
  for (long s = 0; s < batch; ++s) {
    int r = oracle_hyperdiffusion_steps(N, sigma, nsteps, C + s * (size_t)N);
    if (r != OR_OK) {
#pragma omp critical
      if (rc == OR_OK) rc = r;
    }
  }
  return rc;
}

int oracle_batch_ch(int N, int batch, double sigma, double dt_over_dx2, int nsteps, double* C) {
  if (N < 5 || batch < 0) return OR_EINVAL;
  int rc = OR_OK;
#pragma omp parallel for schedule(static)
  for (long s = 0; s < batch; ++s) {
    int r = oracle_ch_steps(N, sigma, dt_over_dx2, nsteps, C + s * (size_t)N);
    if (r != OR_OK) {
#pragma omp critical
      if (rc == OR_OK) rc = r;
    }
  }
  return rc;
}

int oracle_batch_cn(int N, int batch, double sigma_x, int nsteps, double* C) {
  if (N < 5 || batch < 0) return OR_EINVAL;
  int rc = OR_OK;
#pragma omp parallel for schedule(static)
  for (long s = 0; s < batch; ++s) {
    int r = oracle_cn_steps(N, sigma_x, nsteps, C + s * (size_t)N);
    if (r != OR_OK) {
#pragma omp critical
      if (rc == OR_OK) rc = r;
    }
  }
  return rc;
}

/* Per-system tridiagonal bands, each array [batch][N]. */
int oracle_batch_tri(int N, int batch, const double* A, const double* B, const double* Cd,
                     const double* Y, double* U) {
  if (N < 1 || batch < 0) return OR_EINVAL;
  int rc = OR_OK;
#pragma omp parallel for schedule(static)
  for (long s = 0; s < batch; ++s) {
    size_t o = s * (size_t)N;
    int r = oracle_tri_solve(N, A + o, B + o, Cd + o, Y + o, U + o);
    if (r != OR_OK) {
#pragma omp critical
      if (rc == OR_OK) rc = r;
    }
  }
  return rc;
}

"""Pins of the CPU oracle against things other than itself (no GPU needed).

Every check compares the oracle with an independent fact: LAPACK / scipy on the
dense or banded matrix assembled from the band definition, a closed form of
the discrete scheme, an invariant of the scheme, or the convergence order the
cuPentBatch page reports for its exact-solution test (eq. (14), Fig. 2).
"""
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from implicit_pde_stepping_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dense(bands, cyclic):
    """Assemble the N x N matrix: row i holds bands a..e at columns i-2..i+2."""
    bands = np.asarray(bands, dtype=np.float64)
    N = bands.shape[1]
    A = np.zeros((N, N))
    for i in range(N):
        for k in range(5):
            col = i + k - 2
            if cyclic:
                A[i, col % N] += bands[k, i]
            elif 0 <= col < N:
                A[i, col] += bands[k, i]
    return A


def random_dd_bands(N, rng):
    b = rng.uniform(-1, 1, size=(5, N))
    for i in range(N):
        b[2, i] = 1.0 + np.abs(b[[0, 1, 3, 4], i]).sum() + rng.uniform(0, 1)
    return b


def rel(x, ref):
    return np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300)


# ---------------------------------------------------------------------------
# non-cyclic LR solve against LAPACK / scipy
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N", list(range(1, 17)) + [33, 128])
@pytest.mark.parametrize("kind", ["dd", "s0.1", "s1", "s10"])
def test_noncyclic_matches_lapack(N, kind):
    rng = np.random.default_rng(1000 + N)
    bands = random_dd_bands(N, rng) if kind == "dd" else inputs.hyper_bands(N, float(kind[1:]))
    f = rng.uniform(-1, 1, N)
    x = oracle.solve(*bands, f)
    ref = np.linalg.solve(dense(bands, False), f)
    assert rel(x, ref) < 1e-12


def test_noncyclic_config_matrix_matches_solve_banded():
    """N=1024, sigma=1 (the shared-matrix throughput matrix) against scipy's banded LU."""
    N = 1024
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, 8)
    X = oracle.batch_shared(bands, F, cyclic=False)
    ab = np.zeros((5, N))          # scipy's diagonal-ordered form, ab[2 + i - j, j] = A[i, j]
    for k, off in enumerate((-2, -1, 0, 1, 2)):
        # band k of row i sits at column j = i + off -> ab[2 - off, i + off]
        for i in range(N):
            j = i + off
            if 0 <= j < N:
                ab[2 - off, j] = bands[k, i]
    ref = scipy.linalg.solve_banded((2, 2), ab, F)
    assert rel(X, ref) < 1e-12


def test_noncyclic_factor_reproduces_matrix():
    """L R with the factor vectors equals A (L: alpha diag, beta sub, eps subsub; R: unit, gamma, delta)."""
    rng = np.random.default_rng(7)
    N = 12
    bands = random_dd_bands(N, rng)
    alpha, beta, gamma, delta, eps = oracle.factor(*bands)
    Lm = np.diag(alpha) + np.diag(beta[1:], -1) + np.diag(eps[2:], -2)
    Rm = np.eye(N) + np.diag(gamma[:-1], 1) + np.diag(delta[:-2], 2)
    assert np.max(np.abs(Lm @ Rm - dense(bands, False))) < 1e-13


# ---------------------------------------------------------------------------
# cyclic (bordered) solve
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N", list(range(5, 17)) + [64, 257])
@pytest.mark.parametrize("kind", ["dd", "s0.5", "s10.48576"])
def test_cyclic_matches_lapack(N, kind):
    rng = np.random.default_rng(2000 + N)
    bands = random_dd_bands(N, rng) if kind == "dd" else inputs.hyper_bands(N, float(kind[1:]))
    f = rng.uniform(-1, 1, N)
    x = oracle.solve(*bands, f, cyclic=True)
    ref = np.linalg.solve(dense(bands, True), f)
    assert rel(x, ref) < 1e-12


def test_cyclic_rejects_small_n():
    with pytest.raises(oracle.OracleError):
        oracle.solve(*inputs.hyper_bands(4, 1.0), np.ones(4), cyclic=True)


def test_zero_pivot_reported():
    bands = np.zeros((5, 6))
    with pytest.raises(oracle.OracleError):
        oracle.solve(*bands, np.ones(6))


# ---------------------------------------------------------------------------
# manufactured solutions and symmetry
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cyclic", [False, True])
def test_manufactured_solution_persys(cyclic):
    rng = np.random.default_rng(3)
    N, batch = 40, 16
    xs = rng.uniform(-1, 1, (N, batch))
    bands_all = [random_dd_bands(N, rng) for _ in range(batch)]
    for s in range(batch):
        f = dense(bands_all[s], cyclic) @ xs[:, s]
        x = oracle.solve(*bands_all[s], f, cyclic=cyclic)
        assert rel(x, xs[:, s]) < 1e-13


def test_batch_persys_matches_single():
    N, batch = 24, 6
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=3)
    F = inputs.rhs_uniform(N, batch, seed=3).astype(np.float32)
    X = oracle.batch_persys(a, b, c, d, e, F)
    for s in range(batch):
        bands = np.stack([v[:, s].astype(np.float64) for v in (a, b, c, d, e)])
        ref = np.linalg.solve(dense(bands, False), F[:, s].astype(np.float64))
        assert rel(X[:, s], ref) < 1e-12


def test_persymmetry_constant_bands():
    """For symmetric constant bands J A J = A, so reversing f reverses x."""
    N = 301
    bands = inputs.hyper_bands(N, 1.0)
    f = np.random.default_rng(5).uniform(-1, 1, N)
    x = oracle.solve(*bands, f)
    xr = oracle.solve(*bands, f[::-1].copy())
    assert rel(xr[::-1], x) < 1e-13


# ---------------------------------------------------------------------------
# closed forms of the discrete schemes
# ---------------------------------------------------------------------------
def test_hyperdiffusion_discrete_amplification():
    """Periodic Fourier data: each mode k is multiplied by 1/(1 + 16 sigma sin^4(pi k/N)) per step."""
    N, sigma, steps, batch = 512, 0.5, 100, 4
    C0 = inputs.fourier_initial(N, batch)
    CT = oracle.batch_hyperdiffusion(C0, sigma, steps)
    a, b = inputs.fourier_modes(N, batch)
    k = np.arange(1, 9)
    G = 1.0 / (1.0 + 16.0 * sigma * np.sin(np.pi * k / N) ** 4)
    x = np.arange(N) / N
    ph = 2 * np.pi * k[:, None] * x[None, :]
    ref = np.cos(ph).T @ (a * (G ** steps)[:, None]) + np.sin(ph).T @ (b * (G ** steps)[:, None])
    assert rel(CT, ref) < 1e-12
    # the damping is visible: mode 8 loses ~0.46% over 100 steps
    assert abs(G[7] ** steps - 0.99541) < 1e-4


def test_ch_mass_conservation():
    N, batch, steps = 1024, 4, 200
    sigma, k2 = inputs.ch_params(N)
    C0 = inputs.ch_initial(N, batch)
    CT = oracle.batch_ch(C0, sigma, k2, steps)
    assert np.max(np.abs(CT.mean(axis=0) - C0.mean(axis=0))) < 1e-12
    assert np.max(np.abs(CT - C0)) > 1e-6     # it did evolve


def test_ch_linearised_single_mode():
    """Amplitude 1e-7: the cubic term is ~1e-14 relative, so each step multiplies mode k by
    (1 + 4 (dt/dx^2) sin^2(pi k/N)) / (1 + 16 sigma sin^4(pi k/N))."""
    N = 1024
    sigma, k2 = inputs.ch_params(N)
    x = np.arange(N) / N
    for kk, steps in ((3, 20), (40, 20), (71, 20), (200, 2)):
        # steps kept small enough that G^steps >= 1e-3: a mode damped further
        # sinks below the rounding noise of the others
        C0 = 1e-7 * np.cos(2 * np.pi * kk * x)[:, None]
        CT = oracle.batch_ch(C0, sigma, k2, steps)
        s = np.sin(np.pi * kk / N)
        G = (1.0 + 4.0 * k2 * s * s) / (1.0 + 16.0 * sigma * s ** 4)
        assert G ** steps > 1e-3
        assert rel(CT, C0 * G ** steps) < 1e-9


@pytest.mark.parametrize("kk,eps", [(5, 0.5), (60, 0.3), (150, 0.8)])
def test_ch_one_nonlinear_step_closed_form(kk, eps):
    """One step from C = eps cos(theta), theta = 2 pi k x: on the grid cos^3 = (3 cos(theta)
    + cos(3 theta)) / 4 exactly, so C^3 - C has modes k and 3k only, D2 = [1, -2, 1]
    multiplies mode m by -4 sin^2(pi m / N), and the solve divides it by
    1 + 16 sigma sin^4(pi m / N).  The step is therefore a two-mode closed form; the
    cubic shows as the 3k mode, which a dropped or mis-powered cubic would miss."""
    N = 1024
    sigma, k2 = inputs.ch_params(N)
    x = np.arange(N) / N
    th = 2 * np.pi * kk * x
    C0 = (eps * np.cos(th))[:, None]
    C1 = oracle.batch_ch(C0, sigma, k2, 1)
    lam = lambda m: 4.0 * np.sin(np.pi * m / N) ** 2          # noqa: E731
    den = lambda m: 1.0 + 16.0 * sigma * np.sin(np.pi * m / N) ** 4   # noqa: E731
    ak = (eps - k2 * lam(kk) * (0.75 * eps ** 3 - eps)) / den(kk)
    a3k = (-k2 * lam(3 * kk) * 0.25 * eps ** 3) / den(3 * kk)
    ref = ak * np.cos(th) + a3k * np.cos(3 * th)
    assert rel(C1[:, 0], ref) < 1e-12
    assert np.max(np.abs(a3k * np.cos(3 * th))) > 1e-6 * np.max(np.abs(ref))   # the cubic is visible


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_hyperdiffusion_exact_solution_convergence_order():
    """The page's validation set-up (eq. (14), Figs. 1–2): the L2 error against
    A cos(kx) exp(-gamma D k^4 T) falls as N^-2.  Backward Euler with a small
    dt keeps the time error below the spatial one."""
    g = _golden("hyperdiffusion_exact.txt")
    k = 2 * np.pi * g["n"] / g["L"]
    lam = g["gamma"] * g["D"] * k ** 4
    T, dt = g["T"], 1e-9
    steps = int(round(T / dt))
    errs = []
    Ns = (32, 64, 128)
    for N in Ns:
        dx = g["L"] / N
        x = np.arange(N) * dx
        C0 = (g["A"] * np.cos(k * x + g["phi"]))[:, None]
        CT = oracle.batch_hyperdiffusion(C0, g["gamma"] * g["D"] * dt / dx ** 4, steps)[:, 0]
        exact = g["A"] * np.cos(k * x + g["phi"]) * np.exp(-lam * T)
        errs.append(np.sqrt(np.sum((CT - exact) ** 2) * dx))
    orders = [np.log2(errs[i] / errs[i + 1]) for i in range(len(errs) - 1)]
    assert all(abs(o - g["error_order"]) < 0.15 for o in orders), (errs, orders)


# ---------------------------------------------------------------------------
# Crank–Nicolson hyperdiffusion (the page's time scheme, eqs. (5)–(6))
# ---------------------------------------------------------------------------
def test_cn_discrete_amplification():
    """Each periodic Fourier mode k is multiplied per step by
    (1 - 16 sx sin^4(pi k/N)) / (1 + 16 sx sin^4(pi k/N)).  With sx = 10 on
    N = 64 the factor of modes 6..8 is negative (they flip sign every step),
    which a wrong sign in the explicit half would not reproduce."""
    steps, batch = 40, 4
    for N, sx in ((512, 0.5), (64, 10.0)):
        a, b = inputs.fourier_modes(N, batch)
        C0 = inputs.fourier_initial(N, batch)
        k = np.arange(1, 9)
        s4 = np.sin(np.pi * k / N) ** 4
        x = np.arange(N) / N
        ph = 2 * np.pi * k[:, None] * x[None, :]
        CT = oracle.batch_cn(C0, sx, steps)
        G = ((1 - 16 * sx * s4) / (1 + 16 * sx * s4)) ** steps
        ref = np.cos(ph).T @ (a * G[:, None]) + np.sin(ph).T @ (b * G[:, None])
        assert rel(CT, ref) < 1e-12
    assert (1 - 160 * np.sin(np.pi * 6 / 64) ** 4) < 0


def test_cn_conserves_mean_and_matches_one_step_by_hand():
    """The D4 stencil sums to zero, so both halves keep the mean.  One step on
    N = 7 equals a dense solve of the two matrices assembled entry by entry."""
    N, sx = 7, 0.37
    C = np.random.default_rng(11).uniform(-1, 1, N)
    D4 = np.zeros((N, N))
    for i in range(N):
        for off, w in ((-2, 1.0), (-1, -4.0), (0, 6.0), (1, -4.0), (2, 1.0)):
            D4[i, (i + off) % N] += w
    ref = np.linalg.solve(np.eye(N) + sx * D4, (np.eye(N) - sx * D4) @ C)
    got = oracle.batch_cn(C[:, None], sx, 1)[:, 0]
    assert rel(got, ref) < 1e-13
    CT = oracle.batch_cn(inputs.ch_initial(1024, 3), 5.0, 50)
    assert np.max(np.abs(CT.mean(axis=0) - inputs.ch_initial(1024, 3).mean(axis=0))) < 1e-12


def test_cn_exact_solution_second_order():
    """The page's validation (eq. (14), Figs. 1–2) run with its own scheme,
    sigma_x = dt / (2 dx^4): the L2 error against the decaying harmonic falls as
    N^-2.  At fixed N the error against the semi-discrete solution
    (decay rate 16 sin^4(k dx / 2) / dx^4) falls as dt^2: Crank–Nicolson is
    second order in time."""
    g = _golden("hyperdiffusion_exact.txt")
    k = 2 * np.pi * g["n"] / g["L"]
    T = g["T"]

    def err(N, steps, semi_discrete=False):
        dt = T / steps
        dx = g["L"] / N
        x = np.arange(N) * dx
        lam = g["gamma"] * g["D"] * (16 * np.sin(k * dx / 2) ** 4 / dx ** 4 if semi_discrete else k ** 4)
        C0 = (g["A"] * np.cos(k * x + g["phi"]))[:, None]
        CT = oracle.batch_cn(C0, g["gamma"] * g["D"] * dt / (2 * dx ** 4), steps)[:, 0]
        exact = g["A"] * np.cos(k * x + g["phi"]) * np.exp(-lam * T)
        return np.sqrt(np.sum((CT - exact) ** 2) * dx)

    errs = [err(N, 400) for N in (32, 64, 128)]
    orders = [np.log2(errs[i] / errs[i + 1]) for i in range(2)]
    assert all(abs(o - g["error_order"]) < 0.15 for o in orders), (errs, orders)
    et = [err(64, s, semi_discrete=True) for s in (10, 20, 40)]
    t_orders = [np.log2(et[i] / et[i + 1]) for i in range(2)]
    assert all(abs(o - 2.0) < 0.1 for o in t_orders), (et, t_orders)


# ---------------------------------------------------------------------------
# Thomas algorithm (tridiagonal page, section 4.1)
# ---------------------------------------------------------------------------
def tri_dense(a, b, c):
    N = len(b)
    A = np.diag(b).astype(np.float64)
    for i in range(1, N):
        A[i, i - 1] = a[i]
    for i in range(N - 1):
        A[i, i + 1] = c[i]
    return A


@pytest.mark.parametrize("N", list(range(1, 17)) + [33, 200])
@pytest.mark.parametrize("kind", ["dd", "spd"])
def test_thomas_matches_lapack(N, kind):
    """Against LAPACK's banded solver (scipy solve_banded) on diagonally dominant and
    SPD (second-difference) tridiagonal matrices."""
    rng = np.random.default_rng(N)
    if kind == "dd":
        a, c = rng.uniform(-1, 1, N), rng.uniform(-1, 1, N)
        b = 1.0 + np.abs(a) + np.abs(c) + rng.uniform(0, 1, N)
    else:
        a = c = np.full(N, -1.0)
        b = np.full(N, 2.0 + 1e-3)
    y = rng.uniform(-1, 1, N)
    ab = np.zeros((3, N))
    ab[0, 1:] = c[:-1]
    ab[1] = b
    ab[2, :-1] = a[1:]
    ref = scipy.linalg.solve_banded((1, 1), ab, y)
    u = oracle.tri_solve(a, b, c, y)
    assert rel(u, ref) < 1e-11
    # a[0] and c[N-1] are outside the matrix and must be ignored
    a2, c2 = a.copy(), c.copy()
    a2[0], c2[-1] = 123.0, -77.0
    assert np.array_equal(oracle.tri_solve(a2, b, c2, y), u)


def test_thomas_dirichlet_eigenmodes():
    """[-r, 1 + 2r, -r] with the ends truncated has eigenvectors sin(pi j k/(N+1)) and
    eigenvalues 1 + 4 r sin^2(pi k / (2 (N+1))): each mode is divided by its eigenvalue."""
    N, r = 100, 2.5
    j = np.arange(1, N + 1)
    a = c = np.full(N, -r)
    b = np.full(N, 1 + 2 * r)
    for k in (1, 7, 50, 100):
        y = np.sin(np.pi * j * k / (N + 1))
        lam = 1 + 4 * r * np.sin(np.pi * k / (2 * (N + 1))) ** 2
        assert rel(oracle.tri_solve(a, b, c, y), y / lam) < 1e-12


def test_thomas_manufactured_batch_and_zero_pivot():
    N, batch = 77, 9
    a, b, c = inputs.tri_bands(N, batch, seed=4, dtype=np.float64)
    U = inputs.rhs_uniform(N, batch, seed=5)
    Y = np.empty_like(U)
    for s in range(batch):
        Y[:, s] = tri_dense(a[:, s], b[:, s], c[:, s]) @ U[:, s]
    assert rel(oracle.batch_tri(a, b, c, Y), U) < 1e-12
    bz = b.copy()
    bz[0, 3] = 0.0
    with pytest.raises(oracle.OracleError):
        oracle.batch_tri(a, bz, c, Y)

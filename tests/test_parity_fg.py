"""GPU parity: the fixed-grid partitioned shared-matrix solve (pent_fg.cu) against the
CPU oracle and against the TwoSum double-float partitioned kernel, and the fp64 range of
the shared solve: systems scaled by powers of ten from 1e-310 to 1e305, zero systems,
non-finite entries and batches that mix all of them.

The fixed-grid kernel scales every system by the power of two that puts its largest
|f| in [1, 2) before it computes, so its accuracy does not depend on the magnitude of
the data; systems whose largest entry is zero, subnormal, non-finite or beyond the
kernel's exponent window are solved by a native fp64 sweep instead."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F64, dev, host, max_rel_err, random_dd_bands

pytestmark = pytest.mark.gpu


def solve(bands, F, variant="split", cyclic=False, opts=None):
    plan = pent.pent_factor(bands, F.shape[1], cyclic=cyclic)
    if variant != "auto":
        plan.set_variant(variant)
    for k, v in (opts or {}).items():
        plan.set_option(k, v)
    X = dev(F)
    pent.pent_solve(plan, X)
    pent.pent_sync()
    out = host(X)
    assert plan.error() == pent.OK
    plan.close()
    return out


@pytest.mark.parametrize("N", [256, 300, 777, 1024, 1500, 2048])
@pytest.mark.parametrize("batch", [1, 7, 100, 1029])
@pytest.mark.parametrize("sigma", [0.25, 1.0, 10.48576])
def test_fixed_grid_hyper_bands(N, batch, sigma):
    """Constant-band hyperdiffusion matrices, ragged batches (partial system groups) and
    chunk counts from 8 to 64, against the oracle."""
    bands = inputs.hyper_bands(N, sigma)
    F = inputs.rhs_uniform(N, batch, seed=N + batch)
    ref = oracle.batch_shared(bands, F)
    assert max_rel_err(solve(bands, F), ref) < TOL_F64


@pytest.mark.parametrize("N", [256, 513, 1024])
@pytest.mark.parametrize("seed", [1, 2])
def test_fixed_grid_random_bands(N, seed):
    """Random diagonally dominant bands (every row's coefficients different)."""
    rng = np.random.default_rng(seed * 1000 + N)
    bands = random_dd_bands(N, rng)
    F = rng.uniform(-1, 1, (N, 333))
    ref = oracle.batch_shared(bands, F)
    assert max_rel_err(solve(bands, F), ref) < TOL_F64


def test_fixed_grid_matches_twosum_kernel():
    """The same solve by the fixed-grid and by the TwoSum double-float partitioned
    kernels: they agree far inside the tolerance."""
    N, batch = 1024, 2000
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=5)
    a = solve(bands, F)
    b = solve(bands, F, opts={"fixed_grid": 0})
    assert max_rel_err(a, b) < 1e-11
    assert max_rel_err(a, oracle.batch_shared(bands, F)) < TOL_F64


def test_fixed_grid_structured_rhs():
    """Right-hand sides that stress the grid bound: constant, alternating, a single
    spike per system, smooth modes, and the sign pattern of the forward operator's
    largest row of |L^-1 R| (the f that maximises |g|)."""
    N = 1024
    bands = inputs.hyper_bands(N, 1.0)
    cols = [np.ones(N), (-1.0) ** np.arange(N), np.cos(2 * np.pi * 3 * np.arange(N) / N)]
    spike = np.zeros(N)
    spike[500] = 1.0
    cols.append(spike)
    # sign pattern maximising g at row 600: the signs of row 600 of the forward
    # operator L^-1 R (g_i = (f_i - beta_i g_{i-1} - eps_i g_{i-2}) / alpha_i, the
    # oracle's factors), applied to every unit vector at once
    al, be, _, _, ep = oracle.factor(*bands)
    G = np.zeros((N, N))
    for i in range(N):
        G[i] = np.eye(N)[i]
        if i >= 1:
            G[i] -= be[i] * G[i - 1]
        if i >= 2:
            G[i] -= ep[i] * G[i - 2]
        G[i] /= al[i]
    cols.append(np.where(G[600] < 0, -1.0, 1.0))
    F = np.stack(cols, axis=1)
    ref = oracle.batch_shared(bands, F)
    assert max_rel_err(solve(bands, F), ref) < TOL_F64


@pytest.mark.parametrize("variant", ["split", "auto"])
@pytest.mark.parametrize("scale", [1e-310, 1e-300, 1e-40, 1e-35, 1e40, 1e300, 1e305])
def test_shared_solve_fp64_range(variant, scale):
    """Right-hand sides scaled across the fp64 range match the oracle (which solves in
    fp64) to the fp64 tolerance; 1e-310 is subnormal, 1e-300 and 1e305 lie outside the
    scaled kernel's exponent window (native fp64 path)."""
    N, batch = 1024, 640
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=17) * scale
    ref = oracle.batch_shared(bands, F)
    X = solve(bands, F, variant)
    assert np.all(np.isfinite(X))
    assert max_rel_err(X, ref) < TOL_F64


@pytest.mark.parametrize("variant", ["split", "auto"])
def test_shared_solve_mixed_batch(variant):
    """One batch mixing a huge system, a tiny one, a zero one, a subnormal one, systems
    whose entries span 600 orders of magnitude and normal systems: every system matches
    the oracle and the zero system gives exact zeros."""
    N, batch = 1024, 512
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=23)
    F[:, 3] *= 1e300
    F[:, 4] *= 1e-300
    F[:, 5] = 0.0
    F[:, 6] *= 1e-310
    F[:, 7] *= np.logspace(-300, 300, N)
    F[:, 8] *= 1e-35
    F[:, 9] *= 1e40
    F[:100, 10] = 0.0
    X = solve(bands, F, variant)
    assert np.all(X[:, 5] == 0.0)
    ref = oracle.batch_shared(bands, F)
    assert max_rel_err(X, ref) < TOL_F64


def test_shared_solve_non_finite_entries():
    """A system with an inf or NaN entry gives non-finite output in that system only
    (as fp64 arithmetic does); its neighbours are unaffected."""
    N, batch = 512, 64
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=29)
    F[100, 2] = np.inf
    F[200, 3] = np.nan
    X = solve(bands, F)
    assert not np.all(np.isfinite(X[:, 2]))
    assert not np.all(np.isfinite(X[:, 3]))
    keep = [s for s in range(batch) if s not in (2, 3)]
    ref = oracle.batch_shared(bands, F[:, keep])
    assert max_rel_err(X[:, keep], ref) < TOL_F64



def banded_matvec(bands, X, cyclic):
    """A @ X for the [5][N] band array (row i: a_i x_{i-2} + b_i x_{i-1} + c_i x_i +
    d_i x_{i+1} + e_i x_{i+2}); X [N][batch].  Cyclic: the indices wrap around."""
    if cyclic:
        return (bands[0][:, None] * np.roll(X, 2, axis=0) + bands[1][:, None] * np.roll(X, 1, axis=0) +
                bands[2][:, None] * X + bands[3][:, None] * np.roll(X, -1, axis=0) +
                bands[4][:, None] * np.roll(X, -2, axis=0))
    Y = bands[2][:, None] * X
    Y[1:] += bands[1][1:, None] * X[:-1]
    Y[2:] += bands[0][2:, None] * X[:-2]
    Y[:-1] += bands[3][:-1, None] * X[1:]
    Y[:-2] += bands[4][:-2, None] * X[2:]
    return Y


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N", [300, 1024])
def test_outputs_on_binade_edges(cyclic, N):
    """Solutions whose entries are signed powers of two, some moved one ulp below or
    above, so that many outputs fall on or next to a binade edge, where joining a pair
    to fp64 (by integers: a carry into the exponent; by an fp64 add: renormalisation)
    must not lose a factor of two.  x is known exactly; f = A x in fp64 (non-cyclic:
    the fixed-grid kernel; cyclic: the TwoSum partitioned kernel)."""
    rng = np.random.default_rng(17)
    batch = 333
    X = np.ldexp(1.0, rng.integers(-12, 12, (N, batch))) * rng.choice([-1.0, 1.0], (N, batch))
    X[::3] = np.nextafter(X[::3], 0.0)                 # one ulp below the edge
    X[1::7] = np.nextafter(X[1::7], 2.0 * X[1::7])     # one ulp above it
    bands = inputs.hyper_bands(N, 1.0)
    F = banded_matvec(bands, X, cyclic)
    out = solve(bands, F, variant="auto", cyclic=cyclic)
    assert max_rel_err(out, X) < TOL_F64


def test_block_queue_across_solves():
    """The persistent kernel takes every block after a CTA's first from a counter in
    the plan, which the last CTA resets.  One plan solves batches of 1, exactly one
    block per CTA, one block more, several blocks per CTA and a ragged batch in turn:
    a counter left over from an earlier solve would leave blocks unsolved."""
    N = 1024                                  # 32 chunks: CTAs of 8 systems x 32 threads
    bands = inputs.hyper_bands(N, 1.0)
    plan = pent.pent_factor(bands, 4096)
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count   # two CTAs of 8 systems each
    for k, batch in enumerate([1, 16 * sms, 16 * sms + 8, 5000, 37, 16 * sms + 8]):
        F = inputs.rhs_uniform(N, batch, seed=100 + k)
        X = dev(F)
        pent.pent_solve(plan, X)
        pent.pent_sync()
        assert plan.error() == pent.OK
        assert max_rel_err(host(X), oracle.batch_shared(bands, F)) < TOL_F64, batch
    plan.close()

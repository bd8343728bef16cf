"""GPU parity across the fp64 range: every default (AUTO) path of the library against
the CPU oracle, which computes in fp64, on inputs scaled by powers of ten from the
subnormal range to near the top of fp64, and on batches that mix scales.

The double-float kernels scale each system by the power of two that brings its
largest entry into [1, 2) before converting it to pairs of floats, and leave systems
outside their exponent window (zero, subnormal, non-finite, extreme) to native fp64,
so none of these inputs may lose accuracy.  The tolerance is the fp64 one, relative
to each system's largest |x|."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu

SCALES = [1e-310, 1e-300, 1e-40, 1e-35, 1e-8, 1e40, 1e300, 1e305]


def mixed(N, batch, seed):
    """A batch whose systems span the fp64 range: huge, tiny, zero, subnormal,
    600 decades inside one system, a system that is zero on its first rows."""
    F = inputs.rhs_uniform(N, batch, seed=seed)
    F[:, 1] *= 1e300
    F[:, 2] *= 1e-300
    F[:, 3] = 0.0
    F[:, 4] *= 1e-310
    F[:, 5] *= np.logspace(-300, 300, N)
    F[:, 6] *= 1e-35
    F[:, 7] *= 1e40
    F[: N // 3, 8] = 0.0
    return F


def run_solve(bands, F, cyclic):
    plan = pent.pent_factor(bands, F.shape[1], cyclic=cyclic)
    X = dev(F)
    pent.pent_solve(plan, X)
    pent.pent_sync()
    out = host(X)
    assert plan.error() == pent.OK
    plan.close()
    return out


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N", [64, 300, 1024])
@pytest.mark.parametrize("scale", SCALES)
def test_solve_scaled(cyclic, N, scale):
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, 333, seed=N + 1) * scale
    X = run_solve(bands, F, cyclic)
    assert np.all(np.isfinite(X))
    assert max_rel_err(X, oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N", [64, 1024])
def test_solve_mixed_batch(cyclic, N):
    bands = inputs.hyper_bands(N, 2.0)
    F = mixed(N, 200, seed=N)
    X = run_solve(bands, F, cyclic)
    assert np.all(X[:, 3] == 0.0)
    assert max_rel_err(X, oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64


def step(kind, N, C0, nsteps, sigma, k2=0.2):
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), C0.shape[1], cyclic=True)
    C = dev(C0)
    if kind == "hyper":
        pent.hyperdiffusion_step(plan, C, nsteps)
    elif kind == "cn":
        pent.cn_step(plan, C, nsteps)
    else:
        pent.ch_step(plan, C, k2, nsteps)
    pent.pent_sync()
    out = host(C)
    assert plan.error() == pent.OK
    plan.close()
    return out


def step_ref(kind, C0, nsteps, sigma, k2=0.2):
    if kind == "hyper":
        return oracle.batch_hyperdiffusion(C0, sigma, nsteps)
    if kind == "cn":
        return oracle.batch_cn(C0, sigma, nsteps)
    return oracle.batch_ch(C0, sigma, k2, nsteps)


@pytest.mark.parametrize("kind", ["hyper", "cn"])
@pytest.mark.parametrize("nsteps", [1, 6])
@pytest.mark.parametrize("scale", SCALES)
def test_linear_steps_scaled(kind, nsteps, scale):
    """Hyperdiffusion and Crank–Nicolson steps (one launch per step for one step, the
    multi-step kernel for six) on scaled states."""
    N, batch, sigma = 512, 200, 0.7
    C0 = inputs.rhs_uniform(N, batch, seed=7) * scale
    out = step(kind, N, C0, nsteps, sigma)
    assert np.all(np.isfinite(out))
    assert max_rel_err(out, step_ref(kind, C0, nsteps, sigma)) < TOL_F64


@pytest.mark.parametrize("kind", ["hyper", "cn", "ch"])
@pytest.mark.parametrize("nsteps", [1, 6])
def test_steps_mixed_batch(kind, nsteps):
    """States that mix scales in one batch (Cahn–Hilliard keeps its states where the
    explicit cubic stays finite in fp64 over the steps: up to 1e20)."""
    N, batch, sigma = 512, 96, 3.0
    C0 = inputs.rhs_uniform(N, batch, seed=9)
    C0[:, 1] *= 1e300 if kind != "ch" else 1e20
    C0[:, 2] *= 1e-300
    C0[:, 3] = 0.0
    C0[:, 4] *= 1e-310
    C0[:, 5] *= 1e-35
    C0[:, 6] *= 1e40 if kind != "ch" else 1e10
    C0[: N // 3, 7] = 0.0
    out = step(kind, N, C0, nsteps if not (kind == "ch" and nsteps > 1) else 2, sigma)
    ref = step_ref(kind, C0, nsteps if not (kind == "ch" and nsteps > 1) else 2, sigma)
    assert np.all(np.isfinite(ref))
    assert np.all(out[:, 3] == 0.0)
    assert max_rel_err(out, ref) < TOL_F64


@pytest.mark.parametrize("nsteps", [1, 5])
@pytest.mark.parametrize("scale", [1e-310, 1e-300, 1e-40, 1e-35, 1e-8, 0.1, 1e8, 1e15])
def test_ch_steps_scaled(nsteps, scale):
    """Cahn–Hilliard on scaled states where fp64 stays finite: the cubic C^3 becomes
    negligible below about 1e-20 (the scheme is then linear) and dominates above 1;
    states above 2^50 take the native path."""
    N, batch, sigma = 512, 128, 3.0
    C0 = inputs.ch_initial(N, batch, seed=11) * (scale / 0.1)
    ref = step_ref("ch", C0, nsteps, sigma)
    if not np.all(np.isfinite(ref)):
        pytest.skip("the scheme itself overflows fp64 at this scale")
    out = step("ch", N, C0, nsteps, sigma)
    assert max_rel_err(out, ref) < TOL_F64


def test_ch_large_state_native_path():
    """A state of 1e40 (beyond the double-float path's window for the cubic): one
    step matches the oracle."""
    N, batch, sigma = 256, 40, 3.0
    C0 = inputs.ch_initial(N, batch, seed=13) * 1e41
    ref = step_ref("ch", C0, 1, sigma)
    out = step("ch", N, C0, 1, sigma)
    assert np.all(np.isfinite(ref))
    assert max_rel_err(out, ref) < TOL_F64


# ---------------------------------------------------------------------------
# per-system matrices (pent_factor_solve, tri_factor_solve), fp64, AUTO variant
# ---------------------------------------------------------------------------
def persys(bands, F):
    import torch
    N, batch = F.shape
    A = [dev(b) for b in bands]
    X = dev(F)
    info = torch.full((batch,), -1, dtype=torch.int32, device="cuda")
    pent.pent_factor_solve(*A, X, info=info)
    pent.pent_sync()
    assert np.all(host(info) == 0)
    return host(X)


def tri(bands, Y):
    import torch
    N, batch = Y.shape
    A = [dev(b) for b in bands]
    X = dev(Y)
    info = torch.full((batch,), -1, dtype=torch.int32, device="cuda")
    pent.tri_factor_solve(*A, X, info=info)
    pent.pent_sync()
    assert np.all(host(info) == 0)
    return host(X)


@pytest.mark.parametrize("kind", ["pent", "tri"])
@pytest.mark.parametrize("what", ["rhs", "bands", "both"])
@pytest.mark.parametrize("scale", SCALES)
def test_per_system_scaled(kind, what, scale):
    """Right-hand side, matrix or both scaled; the solution scales by scale,
    1/scale or not at all."""
    N, batch = 300, 256
    if kind == "pent":
        bands = list(inputs.persys_bands(N, batch, seed=5, dtype=np.float64))
    else:
        bands = list(inputs.tri_bands(N, batch, seed=5, dtype=np.float64))
    F = inputs.rhs_uniform(N, batch, seed=6)
    if what in ("rhs", "both"):
        F = F * scale
    if what in ("bands", "both"):
        if scale < 1e-300:
            pytest.skip("subnormal matrix entries: fp64's own factorization degenerates")
        bands = [b * scale for b in bands]
    if kind == "pent":
        ref = oracle.batch_persys(*bands, F)
        out = persys(bands, F)
    else:
        ref = oracle.batch_tri(*bands, F)
        out = tri(bands, F)
    if not np.all(np.isfinite(ref)):
        pytest.skip("the solution leaves the fp64 range")
    assert np.all(np.isfinite(out))
    assert max_rel_err(out, ref) < TOL_F64


@pytest.mark.parametrize("kind", ["pent", "tri"])
def test_per_system_mixed_batch(kind):
    """Systems with scaled matrices, scaled right-hand sides, zero and subnormal
    right-hand sides, and rows whose scales span 200 decades inside one system."""
    N, batch = 257, 128
    if kind == "pent":
        bands = [b.copy() for b in inputs.persys_bands(N, batch, seed=8, dtype=np.float64)]
    else:
        bands = [b.copy() for b in inputs.tri_bands(N, batch, seed=8, dtype=np.float64)]
    F = inputs.rhs_uniform(N, batch, seed=9)
    for b in bands:
        b[:, 1] *= 1e300
        b[:, 2] *= 1e-250
        b[:, 7] *= 1e200
    F[:, 3] *= 1e300
    F[:, 4] *= 1e-300
    F[:, 5] = 0.0
    F[:, 6] *= 1e-310
    F[:, 7] *= 1e200
    rowscale = np.logspace(-100, 100, N)
    for b in bands:
        b[:, 8] *= rowscale
    F[:, 8] *= rowscale
    F[: N // 2, 9] = 0.0
    if kind == "pent":
        ref = oracle.batch_persys(*bands, F)
        out = persys(bands, F)
    else:
        ref = oracle.batch_tri(*bands, F)
        out = tri(bands, F)
    assert np.all(out[:, 5] == 0.0)
    assert np.all(np.isfinite(ref))
    assert max_rel_err(out, ref) < TOL_F64


# ---------------------------------------------------------------------------
# systems too long for one CTA (the multi-kernel partitioned form)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("scale", [1e-310, 1e-300, 1e-35, 1e40, 1e300, 1e305])
def test_long_systems_scaled(cyclic, scale):
    N, batch = 5003, 6
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=31) * scale
    X = run_solve(bands, F, cyclic)
    assert np.all(np.isfinite(X))
    assert max_rel_err(X, oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
def test_long_systems_mixed_batch(cyclic):
    N = 5003
    bands = inputs.hyper_bands(N, 1.0)
    F = mixed(N, 10, seed=33)
    X = run_solve(bands, F, cyclic)
    assert np.all(X[:, 3] == 0.0)
    assert max_rel_err(X, oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
def test_long_systems_chunk_scales(cyclic):
    """Systems too long for one CTA scale every chunk by its own power of two: rows
    whose magnitudes differ by hundreds of decades between chunks, a system that is
    zero except for one chunk, a system whose largest entry is subnormal, and one
    with a single subnormal chunk among normal ones."""
    N, batch = 5003, 6
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=35)
    F[:, 0] *= np.repeat(np.logspace(-250, 250, (N + 31) // 32), 32)[:N]   # a scale per chunk
    F[:, 1] = 0.0
    F[2000:2032, 1] = inputs.rhs_uniform(32, 1, seed=36)[:, 0] * 1e-20      # one nonzero chunk
    F[:, 2] *= 1e-312                                                       # subnormal largest entry
    F[1000:1100, 3] *= 1e-320                                               # a subnormal stretch
    F[:, 4] *= 1e306                                                        # above the join's window
    X = run_solve(bands, F, cyclic)
    assert np.all(np.isfinite(X))
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    # the subnormal system: the oracle's own fp64 loses bits on subnormal data, so
    # its reference is the oracle on the data times 2^600 (exact), scaled back (at
    # 1e-312 one subnormal ulp of the output is still only 5e-12 of it)
    ref[:, 2] = np.ldexp(oracle.batch_shared(bands, np.ldexp(F[:, 2:3], 600), cyclic=cyclic)[:, 0], -600)
    assert max_rel_err(X, ref) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
def test_long_systems_non_finite_entry(cyclic):
    """A long system with an inf or NaN entry returns NaN in every entry; the other
    systems of the batch are unaffected."""
    N, batch = 5003, 4
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=37)
    F[1234, 1] = np.inf
    F[4321, 2] = np.nan
    X = run_solve(bands, F, cyclic)
    assert np.all(np.isnan(X[:, 1])) and np.all(np.isnan(X[:, 2]))
    ok = [0, 3]
    assert max_rel_err(X[:, ok], oracle.batch_shared(bands, np.ascontiguousarray(F[:, ok]), cyclic=cyclic)) < TOL_F64

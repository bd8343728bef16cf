"""GPU parity: the partitioned solve of systems too long for one CTA (two-kernel
form: local sweeps, chunk states, periodic border, corrections) against the oracle."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu


def solve(N, batch, sigma, cyclic, seed, variant="auto"):
    bands = inputs.hyper_bands(N, sigma)
    F = inputs.rhs_uniform(N, batch, seed=seed)
    plan = pent.pent_factor(bands, batch, cyclic=cyclic)
    if variant != "auto":
        plan.set_variant(variant)
    X = dev(F)
    l0 = pent.launch_count()
    pent.pent_solve(plan, X)
    pent.pent_sync()
    launches = pent.launch_count() - l0
    out = host(X)
    v = plan.variant(batch)
    plan.close()
    return bands, F, out, launches, v


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N", [2100, 4099, 20000])
@pytest.mark.parametrize("batch", [1, 3, 7, 8, 33])
def test_long_systems_match_oracle(cyclic, N, batch):
    bands, F, out, launches, v = solve(N, batch, 1.0, cyclic, seed=N + batch)
    assert v == pent.VARIANT_SPLIT
    # the local sweeps (with the scales), the chunk states, (the periodic border,) the fix-up
    assert launches == (4 if cyclic else 3)
    assert max_rel_err(out, oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64


@pytest.mark.parametrize("sigma", [0.05, 10.48576])
def test_long_systems_other_sigmas(sigma):
    for cyclic in (False, True):
        bands, F, out, _, v = solve(9000, 16, sigma, cyclic, seed=5)
        assert v == pent.VARIANT_SPLIT
        assert max_rel_err(out, oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64


def test_very_long_systems_sampled():
    """N = 2^20 + 3 rows (32769 chunks), 12 systems: every system against the oracle."""
    N, batch = (1 << 20) + 3, 12
    bands, F, out, _, v = solve(N, batch, 1.0, True, seed=9)
    assert v == pent.VARIANT_SPLIT
    assert max_rel_err(out, oracle.batch_shared(bands, F, cyclic=True)) < TOL_F64


def test_long_plan_repeated_solves_and_batch_growth():
    """The summary buffer grows with the batch; solves stay correct across sizes."""
    N = 5000
    bands = inputs.hyper_bands(N, 1.0)
    plan = pent.pent_factor(bands, 4)
    for batch in (4, 40, 2, 40):
        F = inputs.rhs_uniform(N, batch, seed=batch)
        X = dev(F)
        pent.pent_solve(plan, X)
        pent.pent_sync()
        assert max_rel_err(host(X), oracle.batch_shared(bands, F)) < TOL_F64
    plan.close()


@pytest.mark.parametrize("cyclic", [False, True])
def test_shared_chunk_tables_change_no_bit(cyclic):
    """Interior chunks of a constant-band matrix read one chunk's tables (bitwise equal
    ones, found when the plan is built); the solution is bit-for-bit that of a plan whose
    chunks all read their own tables."""
    N, batch = 40000, 5
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=13)
    out = []
    for dedup in (1, 0):
        plan = pent.pent_factor(bands, batch, cyclic=cyclic)
        plan.set_option("chunk_dedup", dedup)
        X = dev(F)
        pent.pent_solve(plan, X)
        pent.pent_sync()
        out.append(host(X))
        plan.close()
    assert np.array_equal(out[0], out[1])
    assert max_rel_err(out[0], oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64

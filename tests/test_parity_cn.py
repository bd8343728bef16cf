"""GPU parity: Crank–Nicolson hyperdiffusion stepping (cn_step) against the oracle.

The page's time scheme, eqs. (5)–(6): (I + sx D4) C' = (I - sx D4) C with
sx = dt / (2 dx^4), periodic.  Both kernels are checked: the partitioned
double-float kernel (default) and the native one-thread-per-system kernel."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu


def cn_gpu(N, batch, sx, steps, C0, variant="auto"):
    plan = pent.pent_factor(inputs.hyper_bands(N, sx), batch, cyclic=True)
    if variant != "auto":
        plan.set_variant(variant)
    C = dev(C0)
    pent.cn_step(plan, C, steps)
    pent.pent_sync()
    out = host(C)
    plan.close()
    return out


def closed_form(N, batch, sx, steps):
    a, b = inputs.fourier_modes(N, batch)
    k = np.arange(1, 9)
    s4 = np.sin(np.pi * k / N) ** 4
    G = ((1 - 16 * sx * s4) / (1 + 16 * sx * s4)) ** steps
    x = np.arange(N) / N
    ph = 2 * np.pi * k[:, None] * x[None, :]
    return np.cos(ph).T @ (a * G[:, None]) + np.sin(ph).T @ (b * G[:, None])


@pytest.mark.parametrize("variant", ["auto", "thread"])
def test_cn_periodic_workload_full_batch(variant):
    """N=512, dx=1/N, dt/dx^4 = 0.5 (sx = 0.25), batch 4096, Fourier data k=1..8,
    100 steps: oracle on 256 sampled systems, closed form on every system."""
    N, batch, sx, steps = 512, 4096, 0.25, 100
    C0 = inputs.fourier_initial(N, batch)
    out = cn_gpu(N, batch, sx, steps, C0, variant)
    idx = inputs.sample_systems(batch, 256)
    ref = oracle.batch_cn(C0[:, idx], sx, steps)
    assert max_rel_err(out[:, idx], ref) < TOL_F64
    assert max_rel_err(out, closed_form(N, batch, sx, steps)) < 1e-10


@pytest.mark.parametrize("variant", ["auto", "thread"])
def test_cn_sign_flipping_modes(variant):
    """sx = 10 on N = 64: modes 6..8 have negative amplification (they flip sign
    every step), which only a correct explicit half reproduces."""
    N, batch, sx, steps = 64, 40, 10.0, 25
    C0 = inputs.fourier_initial(N, batch)
    out = cn_gpu(N, batch, sx, steps, C0, variant)
    assert max_rel_err(out, oracle.batch_cn(C0, sx, steps)) < TOL_F64
    assert max_rel_err(out, closed_form(N, batch, sx, steps)) < 1e-10


@pytest.mark.parametrize("variant", ["auto", "thread"])
@pytest.mark.parametrize("N", [5, 6, 7, 16, 64, 333, 1000, 2051])
@pytest.mark.parametrize("batch", [1, 100])
def test_cn_ragged(N, batch, variant):
    C0 = inputs.rhs_uniform(N, batch, seed=N + batch)
    out = cn_gpu(N, batch, 0.7, 5, C0, variant)
    assert max_rel_err(out, oracle.batch_cn(C0, 0.7, 5)) < TOL_F64


def test_cn_random_data_large_sigma():
    """Uniform random data keeps every mode; sx = 3e3 on N = 1024 is the stiff
    regime where Crank–Nicolson leaves the highest modes nearly undamped."""
    N, batch, sx, steps = 1024, 64, 3e3, 10
    C0 = inputs.rhs_uniform(N, batch, seed=3)
    out = cn_gpu(N, batch, sx, steps, C0)
    ref = oracle.batch_cn(C0, sx, steps)
    assert max_rel_err(out, ref) < TOL_F64
    assert np.max(np.abs(ref)) > 0.3      # the high modes survive


def test_cn_zero_steps_and_bad_plan():
    N, batch = 16, 4
    C0 = inputs.rhs_uniform(N, batch, seed=1)
    plan = pent.pent_factor(inputs.hyper_bands(N, 1.0), batch, cyclic=True)
    C = dev(C0)
    pent.cn_step(plan, C, 0)
    assert np.array_equal(host(C), C0)
    nc = pent.pent_factor(inputs.hyper_bands(N, 1.0), batch, cyclic=False)
    with pytest.raises(pent.PentError):
        pent.cn_step(nc, C, 1)
    plan.close()
    nc.close()

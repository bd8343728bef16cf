"""GPU parity: periodic hyperdiffusion and Cahn–Hilliard time stepping."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_CH, TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu


def hyper_gpu(N, batch, sigma, steps, C0, variant="auto"):
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
    if variant != "auto":
        plan.set_variant(variant)
    C = dev(C0)
    pent.hyperdiffusion_step(plan, C, steps)
    pent.pent_sync()
    out = host(C)
    plan.close()
    return out


def ch_gpu(N, batch, steps, C0, variant="auto"):
    sigma, k2 = inputs.ch_params(N)
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
    if variant != "auto":
        plan.set_variant(variant)
    C = dev(C0)
    pent.ch_step(plan, C, k2, steps)
    pent.pent_sync()
    out = host(C)
    plan.close()
    return out


def test_hyperdiffusion_workload_full_batch():
    """Cyclic I + 0.5 D4, N=512, batch 4096, Fourier data k=1..8, 100 steps: parity with
    the oracle and with the closed-form discrete amplification per mode."""
    N, batch, sigma, steps = 512, 4096, 0.5, 100
    C0 = inputs.fourier_initial(N, batch)
    out = hyper_gpu(N, batch, sigma, steps, C0)
    ref = oracle.batch_hyperdiffusion(C0, sigma, steps)
    assert max_rel_err(out, ref) < TOL_F64
    a, b = inputs.fourier_modes(N, batch)
    k = np.arange(1, 9)
    G = (1.0 / (1.0 + 16.0 * sigma * np.sin(np.pi * k / N) ** 4)) ** steps
    x = np.arange(N) / N
    ph = 2 * np.pi * k[:, None] * x[None, :]
    exact = np.cos(ph).T @ (a * G[:, None]) + np.sin(ph).T @ (b * G[:, None])
    assert max_rel_err(out, exact) < 1e-10


@pytest.mark.parametrize("N", [5, 6, 7, 64, 333])
@pytest.mark.parametrize("batch", [1, 100])
def test_hyperdiffusion_ragged(N, batch):
    C0 = inputs.rhs_uniform(N, batch, seed=N)
    out = hyper_gpu(N, batch, 0.7, 5, C0)
    ref = oracle.batch_hyperdiffusion(C0, 0.7, 5)
    assert max_rel_err(out, ref) < TOL_F64


def test_ch_workload_2000_steps():
    """Semi-implicit CH, N=1024, batch 16384, gamma=1e-4, dt=0.1 dx^2, 2000 steps:
    parity with the oracle on 256 systems spread over the batch, mass conserved in all."""
    N, batch, steps = 1024, 16384, 2000
    C0 = inputs.ch_initial(N, batch)
    out = ch_gpu(N, batch, steps, C0)
    idx = inputs.sample_systems(batch, 256)
    sigma, k2 = inputs.ch_params(N)
    ref = oracle.batch_ch(C0[:, idx], sigma, k2, steps)
    assert max_rel_err(out[:, idx], ref) < TOL_CH
    assert np.max(np.abs(out.mean(axis=0) - C0.mean(axis=0))) < 1e-12
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("N", [5, 8, 64, 1000])
@pytest.mark.parametrize("batch", [1, 33])
def test_ch_ragged_short(N, batch):
    C0 = inputs.ch_initial(N, batch, seed=N)
    sigma, k2 = 3.0, 0.2
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
    C = dev(C0)
    pent.ch_step(plan, C, k2, 7)
    pent.pent_sync()
    ref = oracle.batch_ch(C0, sigma, k2, 7)
    assert max_rel_err(host(C), ref) < TOL_F64
    plan.close()


def test_ch_linearised_mode_on_gpu():
    N, batch = 1024, 4
    sigma, k2 = inputs.ch_params(N)
    x = np.arange(N) / N
    kk, steps = 40, 20
    C0 = np.repeat((1e-7 * np.cos(2 * np.pi * kk * x))[:, None], batch, axis=1)
    out = ch_gpu(N, batch, steps, C0)
    s = np.sin(np.pi * kk / N)
    G = (1.0 + 4.0 * k2 * s * s) / (1.0 + 16.0 * sigma * s ** 4)
    assert max_rel_err(out, C0 * G ** steps) < 1e-9


def test_zero_steps_is_identity_and_bad_plan_rejected():
    N, batch = 16, 4
    C0 = inputs.ch_initial(N, batch)
    plan = pent.pent_factor(inputs.hyper_bands(N, 1.0), batch, cyclic=True)
    C = dev(C0)
    pent.ch_step(plan, C, 0.1, 0)
    pent.hyperdiffusion_step(plan, C, 0)
    assert np.array_equal(host(C), C0)
    nc = pent.pent_factor(inputs.hyper_bands(N, 1.0), batch, cyclic=False)
    with pytest.raises(pent.PentError):
        pent.ch_step(nc, C, 0.1, 1)
    with pytest.raises(pent.PentError):
        pent.hyperdiffusion_step(nc, C, 1)

"""GPU parity: the persistent multi-step kernel (nsteps >= 2 of hyperdiffusion,
Cahn–Hilliard and Crank–Nicolson in one launch, state kept in registers) against
the oracle, against one launch per step, and its launch count."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu

SIGMA = {"hyper": 0.7, "ch": 3.0, "cn": 0.7}
K2 = 0.2


def run(kind, N, batch, steps, C0, per_step=False, sigma=None, opts=None):
    sigma = SIGMA[kind] if sigma is None else sigma
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
    if per_step:
        plan.set_option("multi_step", 0)
    for k, v in (opts or {}).items():
        plan.set_option(k, v)
    C = dev(C0)
    l0 = pent.launch_count()
    if kind == "hyper":
        pent.hyperdiffusion_step(plan, C, steps)
    elif kind == "ch":
        pent.ch_step(plan, C, K2, steps)
    else:
        pent.cn_step(plan, C, steps)
    pent.pent_sync()
    launches = pent.launch_count() - l0
    out = host(C)
    plan.close()
    return out, launches


def ref(kind, C0, steps, sigma=None):
    sigma = SIGMA[kind] if sigma is None else sigma
    if kind == "hyper":
        return oracle.batch_hyperdiffusion(C0, sigma, steps)
    if kind == "ch":
        return oracle.batch_ch(C0, sigma, K2, steps)
    return oracle.batch_cn(C0, sigma, steps)


def initial(kind, N, batch, seed):
    if kind == "ch":
        return inputs.ch_initial(N, batch, seed=seed)
    return inputs.rhs_uniform(N, batch, seed=seed)


@pytest.mark.parametrize("kind", ["hyper", "ch", "cn"])
@pytest.mark.parametrize("N", [18, 64, 130, 333, 512, 1000, 1024, 2000])
@pytest.mark.parametrize("batch", [1, 33, 100])
def test_multistep_matches_oracle(kind, N, batch):
    steps = 7
    C0 = initial(kind, N, batch, seed=N + batch)
    out, launches = run(kind, N, batch, steps, C0)
    assert max_rel_err(out, ref(kind, C0, steps)) < TOL_F64
    # one launch for all steps where the plan keeps truncated chunk couplings;
    # otherwise (N = 2000: 64 chunks of 32 rows, beyond the one-CTA partitioned
    # cyclic kernel; sigma = 3 with 16-row chunks: couplings decay too slowly to
    # truncate) one solve per step: the fused CH / CN steps in one native launch,
    # hyperdiffusion through the four-launch partitioned solve for long systems
    # (local sweeps, chunk states, periodic border, fix-up)
    assert launches in (1, steps, 4 * steps)
    if kind != "ch" and N <= 1024:
        assert launches == 1
    if N == 2000:
        assert launches == (4 * steps if kind == "hyper" else steps)


@pytest.mark.parametrize("kind", ["hyper", "ch", "cn"])
def test_multistep_equals_one_launch_per_step(kind):
    N, batch, steps = 512, 300, 20
    C0 = initial(kind, N, batch, seed=5)
    a, la = run(kind, N, batch, steps, C0)
    b, lb = run(kind, N, batch, steps, C0, per_step=True)
    assert la == 1 and lb == steps
    assert max_rel_err(a, b) < TOL_F64


@pytest.mark.parametrize("kind", ["hyper", "ch", "cn"])
def test_multistep_more_blocks_than_grid(kind):
    """20000 systems: more blocks of systems than resident CTAs, so the
    persistent grid loops; 256 sampled systems against the oracle."""
    N, batch, steps = 512, 20000, 3
    C0 = initial(kind, N, batch, seed=9)
    out, launches = run(kind, N, batch, steps, C0)
    idx = inputs.sample_systems(batch, 256)
    assert max_rel_err(out[:, idx], ref(kind, C0[:, idx], steps)) < TOL_F64
    assert launches == 1


def test_multistep_hyperdiffusion_closed_form():
    """Config-2 shape: N=512, sigma=0.5, batch 4096, 100 steps in one launch,
    against the discrete amplification factor of every Fourier mode."""
    N, batch, sigma, steps = 512, 4096, 0.5, 100
    C0 = inputs.fourier_initial(N, batch)
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
    C = dev(C0)
    l0 = pent.launch_count()
    pent.hyperdiffusion_step(plan, C, steps)
    pent.pent_sync()
    assert pent.launch_count() - l0 == 1
    out = host(C)
    a, b = inputs.fourier_modes(N, batch)
    k = np.arange(1, 9)
    G = (1.0 / (1.0 + 16.0 * sigma * np.sin(np.pi * k / N) ** 4)) ** steps
    x = np.arange(N) / N
    ph = 2 * np.pi * k[:, None] * x[None, :]
    exact = np.cos(ph).T @ (a * G[:, None]) + np.sin(ph).T @ (b * G[:, None])
    assert max_rel_err(out, exact) < 1e-10
    plan.close()


def test_serial_scan_plans_step_one_launch_at_a_time():
    """With the exact serial chunk scan forced (option serial_chunk_scan) the
    multi-step kernel is not used: one launch per step, same results."""
    N, batch, steps = 333, 40, 4
    C0 = inputs.rhs_uniform(N, batch, seed=2)
    out, launches = run("hyper", N, batch, steps, C0, opts={"serial_chunk_scan": 1})
    assert launches == steps
    assert max_rel_err(out, ref("hyper", C0, steps)) < TOL_F64


@pytest.mark.parametrize("kind", ["ch", "cn", "hyper"])
@pytest.mark.parametrize("steps", [1, 9])
def test_border_correction_skipped_only_where_negligible(kind, steps):
    """Chunks far from the periodic border skip the x_t correction (its E^{-1} G
    entries are below 2^-60 there); the results match plans that apply it in
    every chunk (option border_all_chunks) and the oracle."""
    N, batch = 1024, 64
    C0 = initial(kind, N, batch, seed=21)
    a, _ = run(kind, N, batch, steps, C0)
    b, _ = run(kind, N, batch, steps, C0, opts={"border_all_chunks": 1})
    assert max_rel_err(a, b) < 1e-13
    assert max_rel_err(a, ref(kind, C0, steps)) < TOL_F64


@pytest.mark.parametrize("kind", ["hyper", "ch", "cn"])
@pytest.mark.parametrize("sb", ["8", "16"])
def test_multistep_systems_per_cta(kind, sb):
    """Both CTA shapes of the multi-step kernel (option steps_systems), whatever the
    default for the shape: 8 or 16 systems per CTA give the oracle's result."""
    N, batch, steps = 512, 4100, 4
    C0 = initial(kind, N, batch, seed=31)
    out, launches = run(kind, N, batch, steps, C0, opts={"steps_systems": int(sb)})
    assert launches == 1
    idx = inputs.sample_systems(batch, 200)
    assert max_rel_err(out[:, idx], ref(kind, C0[:, idx], steps)) < TOL_F64


@pytest.mark.parametrize("kind,sigma", [("hyper", 0.5), ("cn", 0.25), ("hyper", 0.05), ("ch", 3.0)])
def test_multistep_low_word_correction_terms(kind, sigma):
    """Where a chunk's responses to its neighbours' states are below 2^-24 in every
    chunk (the first and last 8-row groups when the couplings decay fast), the
    multi-step kernel adds those terms to the low word alone.  Against every term in
    double-float (option cheap_terms = 0) after 50 steps: the same state to 2^-40 of
    max |C|, and both match the oracle."""
    N, batch, steps = 512, 520, 50
    C0 = initial(kind, N, batch, seed=41)
    r = ref(kind, C0, steps, sigma)
    out = []
    for cheap in (1, 0):
        o, launches = run(kind, N, batch, steps, C0, sigma=sigma, opts={"cheap_terms": cheap})
        assert launches == 1
        assert max_rel_err(o, r) < TOL_F64
        out.append(o)
    assert max_rel_err(out[0], out[1]) < 2.0 ** -40

"""GPU parity: shared-matrix solves (pent_factor + pent_solve) against the CPU oracle."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F32, TOL_F64, dev, host, max_rel_err, random_dd_bands

pytestmark = pytest.mark.gpu

VARIANTS_F64 = ["thread", "thread_df", "split"]


def solve_gpu(bands, F, cyclic, variant="auto", dtype="f64", opts=None):
    import torch
    tdt = torch.float64 if dtype == "f64" else torch.float32
    plan = pent.pent_factor(bands, F.shape[1], cyclic=cyclic, dtype=dtype)
    for k, v in (opts or {}).items():
        plan.set_option(k, v)
    if variant != "auto":
        try:
            plan.set_variant(variant)
        except pent.PentError as e:
            plan.close()
            if e.status == pent.ERR_UNSUPPORTED:
                pytest.skip(f"variant {variant} does not exist for N={bands.shape[1]}")
            raise
    X = dev(F, tdt)
    pent.pent_solve(plan, X)
    pent.pent_sync()
    out = host(X)
    plan.close()
    return out


@pytest.mark.parametrize("variant", VARIANTS_F64)
def test_small_workload_full_batch(variant):
    """N=128, batch 1024, sigma=1 non-cyclic, seed 0: one factor + one solve."""
    N, batch = 128, 1024
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=0)
    ref = oracle.batch_shared(bands, F, cyclic=False)
    assert max_rel_err(solve_gpu(bands, F, False, variant), ref) < TOL_F64


@pytest.mark.parametrize("variant", VARIANTS_F64)
@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 9, 17, 64, 100, 257])
@pytest.mark.parametrize("batch", [1, 3, 31, 129, 1000])
def test_ragged_shapes_random_bands(variant, cyclic, N, batch):
    if cyclic and N < 5:
        pytest.skip("cyclic needs N >= 5")
    rng = np.random.default_rng(N * 1000 + batch)
    bands = random_dd_bands(N, rng)
    F = rng.uniform(-1, 1, (N, batch))
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    assert max_rel_err(solve_gpu(bands, F, cyclic, variant), ref) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N,batch", [(5, 7), (64, 200), (1024, 333)])
def test_fp32_plan(cyclic, N, batch):
    rng = np.random.default_rng(11)
    bands = random_dd_bands(N, rng)
    F = rng.uniform(-1, 1, (N, batch)).astype(np.float32)
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    assert max_rel_err(solve_gpu(bands, F, cyclic, dtype="f32"), ref) < TOL_F32


@pytest.mark.parametrize("variant", VARIANTS_F64)
def test_full_size_throughput_workload_sampled(variant):
    """N=1024, batch 65536, sigma=1 (512 MB per array), in the launch configuration the
    benchmark times; 1024 systems spread over the batch are checked against the oracle."""
    N, batch = 1024, 65536
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=0)
    X = solve_gpu(bands, F, False, variant)
    idx = inputs.sample_systems(batch, 1024)
    ref = oracle.batch_shared(bands, F[:, idx], cyclic=False)
    assert max_rel_err(X[:, idx], ref) < TOL_F64
    assert np.all(np.isfinite(X))


@pytest.mark.parametrize("variant", VARIANTS_F64)
@pytest.mark.parametrize("sigma", [0.5, 10.48576])
def test_cyclic_hyper_matrix(variant, sigma):
    N, batch = 1024, 2048
    bands = inputs.hyper_bands(N, sigma)
    F = inputs.rhs_uniform(N, batch, seed=4)
    ref = oracle.batch_shared(bands, F, cyclic=True)
    assert max_rel_err(solve_gpu(bands, F, True, variant), ref) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("scale", [1e-25, 1e-8, 1e8, 1e25])
def test_df_dynamic_range_scaled_rhs(cyclic, scale):
    """The double-float kernel keeps fp64-class relative accuracy across magnitudes."""
    N, batch = 200, 300
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=8) * scale
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    assert max_rel_err(solve_gpu(bands, F, cyclic, "thread_df"), ref) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
def test_df_zero_and_spike_systems(cyclic):
    """Zero right-hand sides give (near) zero; single spikes and mixed scales stay accurate."""
    N, batch = 96, 64
    bands = inputs.hyper_bands(N, 2.0)
    F = inputs.rhs_uniform(N, batch, seed=3)
    F[:, 0] = 0.0
    F[:, 1] = 0.0
    F[17, 1] = 1.0
    F[:, 2] *= 1e-12
    F[40:, 3] = 0.0
    X = solve_gpu(bands, F, cyclic, "thread_df")
    assert np.max(np.abs(X[:, 0])) < 1e-30
    ref = oracle.batch_shared(bands, F[:, 1:], cyclic=cyclic)
    assert max_rel_err(X[:, 1:], ref) < TOL_F64


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N,sigma", [(1024, 1e4), (300, 50.0), (1024, 1.0)])
def test_split_serial_and_parallel_scans(cyclic, N, sigma):
    """The partitioned kernel with its parallel (truncated-coupling) scan and with the
    exact serial scan forced; sigma = 1e4 couples chunks too strongly for truncation,
    so the plan itself falls back to the serial scan there."""
    bands = inputs.hyper_bands(N, sigma)
    F = inputs.rhs_uniform(N, 96, seed=N)
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    assert max_rel_err(solve_gpu(bands, F, cyclic, "split"), ref) < TOL_F64
    assert max_rel_err(solve_gpu(bands, F, cyclic, "split", opts={"serial_chunk_scan": 1}),
                       ref) < TOL_F64


def test_zero_pivot_is_reported():
    bands = np.zeros((5, 16))
    with pytest.raises(pent.PentError) as ei:
        pent.pent_factor(bands, 4)
    assert ei.value.status == pent.ERR_ZERO_PIVOT


def test_singular_border_is_reported():
    # last two rows/columns decoupled (G = H = 0) and B = [[1, 1], [1, 1]]:
    # B - H^T E^{-1} G = B is exactly singular.
    N = 16
    bands = inputs.hyper_bands(N, 1.0)
    for k, i in ((0, 0), (1, 0), (0, 1), (4, N - 4), (3, N - 3), (4, N - 3),
                 (0, N - 2), (1, N - 2), (4, N - 2), (0, N - 1), (3, N - 1), (4, N - 1)):
        bands[k, i] = 0.0
    bands[2, N - 2] = bands[3, N - 2] = bands[1, N - 1] = bands[2, N - 1] = 1.0
    with pytest.raises(pent.PentError) as ei:
        pent.pent_factor(bands, 4, cyclic=True)
    assert ei.value.status == pent.ERR_ZERO_PIVOT


def test_solve_argument_errors():
    import torch
    plan = pent.pent_factor(inputs.hyper_bands(8, 1.0), 4)
    with pytest.raises(ValueError):
        pent.pent_solve(plan, torch.zeros(7, 4, dtype=torch.float64, device="cuda"))
    with pytest.raises(TypeError):
        pent.pent_solve(plan, torch.zeros(8, 4, dtype=torch.float32, device="cuda"))
    base = torch.zeros(8 * 5 + 1, dtype=torch.float64, device="cuda")
    mis = base[1:].view(8, 5)       # 8-byte but not 16-byte aligned
    st = pent.lib().pent_solve(plan.handle, __import__("ctypes").c_void_p(mis.data_ptr()), 5, None)
    assert st == pent.ERR_INVALID_ARG
    plan.close()


def test_batch_smaller_than_plan_and_stream_order():
    import torch
    N = 300
    bands = inputs.hyper_bands(N, 2.0)
    plan = pent.pent_factor(bands, 4096)
    F = inputs.rhs_uniform(N, 77, seed=9)
    s = torch.cuda.Stream()
    X = dev(F)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        pent.pent_solve(plan, X, stream=s)
        pent.pent_solve(plan, X, stream=s)      # two solves in order on one stream
    s.synchronize()
    ref = oracle.batch_shared(bands, oracle.batch_shared(bands, F), cyclic=False)
    assert max_rel_err(host(X), ref) < TOL_F64


@pytest.mark.parametrize("sigma", [0.05, 1.0, 50.0])
@pytest.mark.parametrize("N", [64, 1000, 2051])
def test_cyclic_twisted_border_reach(sigma, N):
    """The twisted kernel applies the periodic-border terms only in the rows near the
    two ends where they exceed 2^-60 (few rows for small sigma, all rows for large):
    parity with the oracle on random right-hand sides."""
    batch = 512
    bands = inputs.hyper_bands(N, sigma)
    F = inputs.rhs_uniform(N, batch, seed=N)
    ref = oracle.batch_shared(bands, F, cyclic=True)
    plan = pent.pent_factor(bands, batch, cyclic=True)
    plan.set_variant("thread_df")
    X = dev(F)
    pent.pent_solve(plan, X)
    assert max_rel_err(host(X), ref) < TOL_F64
    plan.close()


@pytest.mark.parametrize("depth", ["0", "4", "8", "12"])
@pytest.mark.parametrize("cyclic", [False, True])
def test_twisted_prefetch_depths(depth, cyclic):
    """The twisted kernel's cp.async ring depths other than the default 6, and the
    register-ring kernel (ring depth 0), against the oracle."""
    N, batch = 700, 1024
    bands = inputs.hyper_bands(N, 0.9)
    F = inputs.rhs_uniform(N, batch, seed=int(depth) + 1)
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    assert max_rel_err(solve_gpu(bands, F, cyclic, "thread_df", opts={"twisted_ring": int(depth)}),
                       ref) < TOL_F64


@pytest.mark.parametrize("variant", VARIANTS_F64)
@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("N", [300, 1024, 4099])
def test_weakly_dominant_hyperdiffusion_matrix(variant, cyclic, N):
    """sigma = 1000: I + sigma D4 is barely more than sigma D4, the eliminated
    couplings decay slowly (chunk couplings too slow to truncate, so the exact
    scans and wide border reaches are exercised); condition ~1.6e4."""
    batch = 256
    bands = inputs.hyper_bands(N, 1000.0)
    F = inputs.rhs_uniform(N, batch, seed=N + 7)
    ref = oracle.batch_shared(bands, F, cyclic=cyclic)
    assert max_rel_err(solve_gpu(bands, F, cyclic, variant), ref) < TOL_F64

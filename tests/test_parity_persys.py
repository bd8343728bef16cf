"""GPU parity: per-system factor + solve (pent_factor_solve) against the CPU oracle."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F32, TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu


def run_gpu(bands, F, dtype, info=True):
    import torch
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    dB = [dev(v, tdt) for v in bands]
    X = dev(F, tdt)
    inf = torch.full((F.shape[1],), -1, dtype=torch.int32, device="cuda") if info else None
    pent.pent_factor_solve(*dB, X, info=inf)
    pent.pent_sync()
    return host(X), (host(inf) if info else None), [host(b) for b in dB]


@pytest.mark.parametrize("dtype,tol", [(np.float32, TOL_F32), (np.float64, TOL_F64)])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 33, 256])
@pytest.mark.parametrize("batch", [1, 5, 127, 1000])
def test_ragged_shapes(dtype, tol, N, batch):
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=N + batch, dtype=dtype)
    F = inputs.rhs_uniform(N, batch, seed=N + batch).astype(dtype)
    ref = oracle.batch_persys(a, b, c, d, e, F)
    X, info, bands_after = run_gpu((a, b, c, d, e), F, dtype)
    assert max_rel_err(X, ref) < tol
    assert np.all(info == 0)
    for before, after in zip((a, b, c, d, e), bands_after):   # bands are left unchanged
        assert np.array_equal(before, after)


def test_full_size_fp32_workload_sampled():
    """N=256, batch 262144, fp32, strictly diagonally dominant per-system bands."""
    N, batch = 256, 262144
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=0)
    F = inputs.rhs_uniform(N, batch, seed=0).astype(np.float32)
    X, info, _ = run_gpu((a, b, c, d, e), F, np.float32)
    idx = inputs.sample_systems(batch, 2048)
    ref = oracle.batch_persys(a[:, idx], b[:, idx], c[:, idx], d[:, idx], e[:, idx], F[:, idx])
    assert max_rel_err(X[:, idx], ref) < TOL_F32
    assert np.all(info == 0)
    assert np.all(np.isfinite(X))


def test_zero_pivot_reported_per_system():
    N, batch = 10, 4
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=1, dtype=np.float64)
    c[0, 1] = 0.0          # system 1: alpha_1 = c_1 = 0 -> info 1
    a[:, 2] = b[:, 2] = d[:, 2] = e[:, 2] = 0.0
    c[6, 2] = 0.0          # system 2: diagonal matrix with a zero at row 7 -> info 7
    F = inputs.rhs_uniform(N, batch, seed=1)
    X, info, _ = run_gpu((a, b, c, d, e), F, np.float64)
    assert list(info) == [0, 1, 7, 0]
    ok = [0, 3]
    ref = oracle.batch_persys(a[:, ok], b[:, ok], c[:, ok], d[:, ok], e[:, ok], F[:, ok])
    assert max_rel_err(X[:, ok], ref) < TOL_F64


def test_work_too_small_rejected():
    import torch
    N, batch = 16, 8
    bands = [torch.ones(N, batch, dtype=torch.float64, device="cuda") for _ in range(5)]
    X = torch.ones(N, batch, dtype=torch.float64, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        pent.pent_factor_solve(*bands, X, work=small)

"""GPU parity: pent_solve_host (right-hand sides and solutions in host memory,
copies overlapped with the solves) against the oracle."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F32, TOL_F64, max_rel_err

pytestmark = pytest.mark.gpu


def pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("batch,chunks", [(1, 0), (100, 3), (1000, 8), (4097, 5), (20000, 0)])
def test_solve_host_matches_oracle(cyclic, batch, chunks):
    N = 300
    bands = inputs.hyper_bands(N, 0.8)
    F = inputs.rhs_uniform(N, batch, seed=batch)
    plan = pent.pent_factor(bands, batch, cyclic=cyclic)
    X = pent.pent_solve_host(plan, pinned(F), chunks=chunks)
    pent.pent_sync()
    assert max_rel_err(X.numpy(), oracle.batch_shared(bands, F, cyclic=cyclic)) < TOL_F64
    plan.close()


def test_solve_host_in_place_repeated_and_fp32():
    N, batch = 128, 5000
    bands = inputs.hyper_bands(N, 1.0)
    plan = pent.pent_factor(bands, batch)
    H = pinned(inputs.rhs_uniform(N, batch, seed=1))
    ref = oracle.batch_shared(bands, H.numpy().copy())
    for _ in range(3):                           # same buffers, calls ordered on one stream
        G = pinned(inputs.rhs_uniform(N, batch, seed=1))
        pent.pent_solve_host(plan, G, G, chunks=4)   # in place
    pent.pent_sync()
    assert max_rel_err(G.numpy(), ref) < TOL_F64
    plan.close()
    p32 = pent.pent_factor(bands, batch, dtype="f32")
    F32 = inputs.rhs_uniform(N, batch, seed=2).astype(np.float32)
    X = pent.pent_solve_host(p32, pinned(F32), chunks=6)
    pent.pent_sync()
    assert max_rel_err(X.numpy(), oracle.batch_shared(bands, F32)) < TOL_F32
    p32.close()


def test_solve_host_full_headline_size_sampled():
    """N = 1024, batch 65536 (the bench shape) through the host path; 256 sampled systems."""
    N, batch = 1024, 65536
    bands = inputs.hyper_bands(N, 1.0)
    F = inputs.rhs_uniform(N, batch, seed=0)
    plan = pent.pent_factor(bands, batch)
    X = pent.pent_solve_host(plan, pinned(F))
    pent.pent_sync()
    idx = inputs.sample_systems(batch, 256)
    assert max_rel_err(X.numpy()[:, idx], oracle.batch_shared(bands, F[:, idx])) < TOL_F64
    plan.close()

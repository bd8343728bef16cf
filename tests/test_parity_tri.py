"""GPU parity: batched tridiagonal solves (tri_factor_solve) against the oracle's
Thomas algorithm, both kernels (one thread per system; partitioned fp32), and
periodic implicit diffusion through a pentadiagonal plan with a = e = 0."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F32, TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu

CASES = [("thread", np.float64, TOL_F64), ("thread", np.float32, TOL_F32),
         ("split", np.float32, TOL_F32), ("thread_df", np.float64, TOL_F64), ("auto", np.float32, TOL_F32),
         ("auto", np.float64, TOL_F64)]


def run(variant, dtype, N, batch, seed, bz=None):
    import torch
    a, b, c = inputs.tri_bands(N, batch, seed=seed, dtype=dtype)
    if bz is not None:
        b = b.copy()
        b[bz] = 0
    y = inputs.rhs_uniform(N, batch, seed=seed + 1).astype(dtype)
    X = dev(y)
    info = torch.zeros(batch, dtype=torch.int32, device="cuda")
    pent.tri_factor_solve(dev(a), dev(b), dev(c), X, variant=variant, info=info)
    pent.pent_sync()
    return (a, b, c, y), host(X), host(info)


@pytest.mark.parametrize("variant,dtype,tol", CASES, ids=[f"{v}-{d.__name__}" for v, d, _ in CASES])
@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 9, 16, 17, 100, 255, 256, 257, 300, 512])
@pytest.mark.parametrize("batch", [1, 33, 1000])
def test_tri_matches_oracle(variant, dtype, tol, N, batch):
    (a, b, c, y), x, info = run(variant, dtype, N, batch, seed=N + batch)
    assert not info.any()
    assert max_rel_err(x, oracle.batch_tri(a, b, c, y)) < tol


@pytest.mark.parametrize("dtype,tol", [(np.float64, TOL_F64), (np.float32, TOL_F32)])
@pytest.mark.parametrize("N", [513, 1000, 4099])
def test_tri_thread_large_n(dtype, tol, N):
    (a, b, c, y), x, info = run("auto", dtype, N, 70, seed=N)
    assert not info.any()
    assert max_rel_err(x, oracle.batch_tri(a, b, c, y)) < tol


@pytest.mark.parametrize("variant", ["split", "thread"])
def test_tri_full_size_fp32_sampled(variant):
    """N = 256, batch 262144, fp32 (the per-system workload shape): 256 sampled systems."""
    N, batch = 256, 262144
    (a, b, c, y), x, info = run(variant, np.float32, N, batch, seed=0)
    assert not info.any()
    idx = inputs.sample_systems(batch, 256)
    ref = oracle.batch_tri(a[:, idx], b[:, idx], c[:, idx], y[:, idx])
    assert max_rel_err(x[:, idx], ref) < TOL_F32


@pytest.mark.parametrize("variant,dtype", [("thread", np.float64), ("split", np.float32),
                                           ("thread", np.float32), ("thread_df", np.float64)])
def test_tri_zero_pivot_reported(variant, dtype):
    """b_0 = 0 in system 3 (a zero first pivot for every elimination order that starts
    there): info flags system 3 only; the other systems are solved."""
    N, batch = 64, 40
    (a, b, c, y), x, info = run(variant, dtype, N, batch, seed=2, bz=(0, 3))
    assert info[3] != 0
    assert np.count_nonzero(info) == 1
    keep = np.array([s for s in range(batch) if s != 3])
    ref = oracle.batch_tri(a[:, keep], b[:, keep], c[:, keep], y[:, keep])
    assert max_rel_err(x[:, keep], ref) < (TOL_F64 if dtype == np.float64 else TOL_F32)


def test_tri_argument_errors():
    import torch
    N, batch = 16, 4
    z = torch.zeros((N, batch), dtype=torch.float64, device="cuda")
    with pytest.raises(pent.PentError):            # the partitioned kernel is fp32 only
        pent.tri_factor_solve(z, z, z, z.clone(), variant="split")
    z32 = torch.zeros((1024, batch), dtype=torch.float32, device="cuda")
    with pytest.raises(pent.PentError):            # ... and N <= 512
        pent.tri_factor_solve(z32, z32, z32, z32.clone(), variant="split")
    z16 = torch.zeros((N, batch), dtype=torch.float32, device="cuda")
    with pytest.raises(pent.PentError):            # the double-float kernel is for fp64 systems
        pent.tri_factor_solve(z16, z16, z16, z16.clone(), variant="thread_df")


def test_periodic_implicit_diffusion_through_pentadiagonal_plan():
    """(I - r D2) u^{n+1} = u^n, periodic: a pentadiagonal cyclic plan with a = e = 0
    and bands [-r, 1 + 2r, -r] divides Fourier mode k by 1 + 4 r sin^2(pi k / N) per step."""
    N, batch, r, steps = 256, 512, 3.0, 20
    bands = np.zeros((5, N))
    bands[1], bands[2], bands[3] = -r, 1 + 2 * r, -r
    plan = pent.pent_factor(bands, batch, cyclic=True)
    C0 = inputs.fourier_initial(N, batch)
    C = dev(C0)
    pent.hyperdiffusion_step(plan, C, steps)
    out = host(C)
    plan.close()
    a, b = inputs.fourier_modes(N, batch)
    k = np.arange(1, 9)
    G = (1.0 / (1.0 + 4 * r * np.sin(np.pi * k / N) ** 2)) ** steps
    x = np.arange(N) / N
    ph = 2 * np.pi * k[:, None] * x[None, :]
    exact = np.cos(ph).T @ (a * G[:, None]) + np.sin(ph).T @ (b * G[:, None])
    assert max_rel_err(out, exact) < 1e-10


def to_blocked(x, bs):
    """Interleaved [N][batch] -> block-interleaved [batch / bs][N][bs]."""
    N, batch = x.shape
    return np.ascontiguousarray(x.reshape(N, batch // bs, bs).transpose(1, 0, 2))


def from_blocked(x):
    nb, N, bs = x.shape
    return np.ascontiguousarray(x.transpose(1, 0, 2).reshape(N, nb * bs))


@pytest.mark.parametrize("variant,dtype,tol", CASES[:4], ids=[f"{v}-{d.__name__}" for v, d, _ in CASES[:4]])
@pytest.mark.parametrize("bs", [16, 32, 8, 48])
@pytest.mark.parametrize("N", [7, 256, 300])
def test_tri_block_interleaved(variant, dtype, tol, bs, N):
    """The page's block-interleaved layout (blocks of bs systems, each an interleaved
    [N][bs] array): same solutions as the oracle.  bs = 8 is not a multiple of 16, so
    the partitioned kernel stages rows with cp.async instead of tensor maps."""
    import torch
    batch = bs * 9
    a, b, c = inputs.tri_bands(N, batch, seed=N + bs, dtype=dtype)
    y = inputs.rhs_uniform(N, batch, seed=N + bs + 1).astype(dtype)
    ref = oracle.batch_tri(a, b, c, y)
    X = dev(to_blocked(y, bs))
    info = torch.zeros(batch, dtype=torch.int32, device="cuda")
    pent.tri_factor_solve(dev(to_blocked(a, bs)), dev(to_blocked(b, bs)), dev(to_blocked(c, bs)), X,
                          variant=variant, info=info, block_size=bs)
    pent.pent_sync()
    assert not host(info).any()
    assert max_rel_err(from_blocked(host(X)), ref) < tol


def test_tri_block_size_must_divide_batch():
    import torch
    z = torch.zeros((16, 4), dtype=torch.float32, device="cuda")
    work = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    L = pent.lib()
    p = [ctypes_ptr(z) for _ in range(4)]
    assert L.tri_factor_solve(*p, 4, 16, pent.F32, pent.VARIANT_THREAD, 3, ctypes_ptr(work), 1 << 16, None,
                              None) == pent.ERR_INVALID_ARG


def ctypes_ptr(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("variant", ["split", "thread"])
@pytest.mark.parametrize("N", [64, 256, 300, 512])
def test_tri_weakly_dominant(variant, N):
    """Second-difference systems [-1, 2 + eps, -1] (eps in [0.1, 0.2]): the
    eliminated couplings decay slowly (factor ~0.7 per row), so a chunk's boundary
    terms reach far into its neighbours; the partitioned kernel's interface must be
    exact, not merely dominated."""
    batch = 96
    rng = np.random.default_rng(N)
    eps = rng.uniform(0.1, 0.2, batch).astype(np.float32)
    a = np.full((N, batch), -1.0, np.float32)
    c = np.full((N, batch), -1.0, np.float32)
    a[0] = 0.0
    c[-1] = 0.0
    b = (2.0 + eps)[None, :].repeat(N, axis=0).astype(np.float32)
    y = inputs.rhs_uniform(N, batch, seed=N).astype(np.float32)
    X = dev(y)
    pent.tri_factor_solve(dev(a), dev(b), dev(c), X, variant=variant)
    pent.pent_sync()
    assert max_rel_err(host(X), oracle.batch_tri(a, b, c, y)) < TOL_F32


def test_tri_fp64_double_float_matches_native():
    """fp64 systems: the double-float kernel (the fp64 default) and the native one agree with
    the oracle at N = 256, batch 65536 (1024 sampled systems)."""
    N, batch = 256, 65536
    for variant in ("thread_df", "thread"):
        (a, b, c, y), x, info = run(variant, np.float64, N, batch, seed=5)
        assert not info.any()
        idx = inputs.sample_systems(batch, 1024)
        ref = oracle.batch_tri(a[:, idx], b[:, idx], c[:, idx], y[:, idx])
        assert max_rel_err(x[:, idx], ref) < TOL_F64

"""GPU parity: per-system factor + solve (pent_factor_solve) against the CPU oracle, both
kernels (one thread per system; partitioned fp32 with TMA tiles) and the automatic choice."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F32, TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu

CASES = [("auto", np.float64, TOL_F64), ("thread", np.float64, TOL_F64), ("thread", np.float32, TOL_F32),
         ("split", np.float32, TOL_F32), ("auto", np.float32, TOL_F32)]
IDS = [f"{v}-{d.__name__}" for v, d, _ in CASES]


def run_gpu(bands, F, dtype, info=True, variant="auto"):
    import torch
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    dB = [dev(v, tdt) for v in bands]
    X = dev(F, tdt)
    inf = torch.full((F.shape[1],), -1, dtype=torch.int32, device="cuda") if info else None
    pent.pent_factor_solve(*dB, X, info=inf, variant=variant)
    pent.pent_sync()
    return host(X), (host(inf) if info else None), [host(b) for b in dB]


@pytest.mark.parametrize("variant,dtype,tol", CASES, ids=IDS)
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 15, 16, 17, 33, 100, 255, 256, 257, 300, 512])
@pytest.mark.parametrize("batch", [1, 5, 127, 1000])
def test_ragged_shapes(variant, dtype, tol, N, batch):
    """batch 1000 takes the TMA-tile path of the split kernel (row pitch a multiple of 16 bytes),
    1, 5 and 127 its per-thread cp.async path; N spans one to 32 chunks with ragged tails."""
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=N + batch, dtype=dtype)
    F = inputs.rhs_uniform(N, batch, seed=N + batch).astype(dtype)
    ref = oracle.batch_persys(a, b, c, d, e, F)
    X, info, bands_after = run_gpu((a, b, c, d, e), F, dtype, variant=variant)
    assert max_rel_err(X, ref) < tol
    assert np.all(info == 0)
    for before, after in zip((a, b, c, d, e), bands_after):   # bands are left unchanged
        assert np.array_equal(before, after)


@pytest.mark.parametrize("variant", ["split", "thread"])
def test_full_size_fp32_workload_sampled(variant):
    """N=256, batch 262144, fp32, strictly diagonally dominant per-system bands."""
    N, batch = 256, 262144
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=0)
    F = inputs.rhs_uniform(N, batch, seed=0).astype(np.float32)
    X, info, _ = run_gpu((a, b, c, d, e), F, np.float32, variant=variant)
    idx = inputs.sample_systems(batch, 2048)
    ref = oracle.batch_persys(a[:, idx], b[:, idx], c[:, idx], d[:, idx], e[:, idx], F[:, idx])
    assert max_rel_err(X[:, idx], ref) < TOL_F32
    assert np.all(info == 0)
    assert np.all(np.isfinite(X))


@pytest.mark.parametrize("variant,dtype,tol", CASES, ids=IDS)
@pytest.mark.parametrize("N", [64, 256, 300, 512])
def test_weakly_dominant(variant, dtype, tol, N):
    """[1, -4, 6 + eps, -4, 1] with eps in [0.1, 0.2] per system (condition ~100): the
    couplings between chunks decay slowly, so an inexact chunk interface would show."""
    batch = 512
    rng = np.random.default_rng(N)
    eps = rng.uniform(0.1, 0.2, batch)
    one = np.ones((N, batch))
    a, b, c, d, e = (one, -4 * one, (6 + eps) * one, -4 * one, one)
    a, b, c, d, e = (v.astype(dtype) for v in (a, b, c, d, e))
    F = inputs.rhs_uniform(N, batch, seed=N).astype(dtype)
    ref = oracle.batch_persys(a, b, c, d, e, F)
    X, info, _ = run_gpu((a, b, c, d, e), F, dtype, variant=variant)
    assert np.all(info == 0)
    assert max_rel_err(X, ref) < tol


@pytest.mark.parametrize("variant,dtype", [("thread", np.float64), ("thread_df", np.float64),
                                           ("thread", np.float32), ("split", np.float32)])
def test_zero_pivot_reported_per_system(variant, dtype):
    N, batch = 40, 5
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=1, dtype=dtype)
    c[0, 1] = 0.0          # system 1: alpha_1 = c_1 = 0 -> info 1
    for s, row in ((2, 6), (4, 20)):
        a[:, s] = b[:, s] = d[:, s] = e[:, s] = 0.0
        c[row, s] = 0.0    # diagonal matrix with a zero at row row + 1 (second chunk for system 4)
    F = inputs.rhs_uniform(N, batch, seed=1).astype(dtype)
    X, info, _ = run_gpu((a, b, c, d, e), F, dtype, variant=variant)
    assert list(info) == [0, 1, 7, 0, 21]
    ok = [0, 3]
    ref = oracle.batch_persys(a[:, ok], b[:, ok], c[:, ok], d[:, ok], e[:, ok], F[:, ok])
    assert max_rel_err(X[:, ok], ref) < (TOL_F64 if dtype == np.float64 else TOL_F32)


def test_split_variant_limits():
    import torch
    for N, tdt, v in ((16, torch.float64, "split"), (513, torch.float32, "split"),
                      (16, torch.float32, "thread_df")):
        bands = [torch.ones(N, 8, dtype=tdt, device="cuda") for _ in range(5)]
        X = torch.ones(N, 8, dtype=tdt, device="cuda")
        with pytest.raises(pent.PentError) as ex:
            pent.pent_factor_solve(*bands, X, variant=v)
        assert ex.value.status == pent.ERR_UNSUPPORTED


@pytest.mark.parametrize("scale", [1e-25, 1e-8, 1e8, 1e25])
def test_fp64_double_float_dynamic_range(scale):
    """The double-float fp64 kernel keeps fp64-class relative accuracy when the bands and
    the right-hand side sit far from 1 (scaled alike, so the pivots, their reciprocals and
    the intermediate values span 1e-25..1e25 while the solution stays O(1))."""
    N, batch = 300, 257
    a, b, c, d, e = (v * scale for v in inputs.persys_bands(N, batch, seed=7, dtype=np.float64))
    F = inputs.rhs_uniform(N, batch, seed=7) * scale
    ref = oracle.batch_persys(a, b, c, d, e, F)
    X, info, _ = run_gpu((a, b, c, d, e), F, np.float64, variant="thread_df")
    assert np.all(info == 0)
    assert max_rel_err(X, ref) < TOL_F64


def test_split_needs_no_work_buffer():
    """Through the C ABI: the split kernel accepts a NULL work buffer; the thread kernel
    rejects it before queueing anything."""
    import ctypes
    import torch
    L = pent.lib()
    N, batch = 64, 32
    bands = [dev(v) for v in inputs.persys_bands(N, batch, seed=3)]
    F = inputs.rhs_uniform(N, batch, seed=3).astype(np.float32)
    X = dev(F)
    vp = [ctypes.c_void_p(t.data_ptr()) for t in bands]
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.pent_factor_solve_ex(*vp, ctypes.c_void_p(X.data_ptr()), N, batch, pent.F32,
                                  pent.VARIANT_THREAD, 0, None, 0, None, st) == pent.ERR_INVALID_ARG
    assert np.array_equal(host(X), F)
    assert L.pent_factor_solve_ex(*vp, ctypes.c_void_p(X.data_ptr()), N, batch, pent.F32,
                                  pent.VARIANT_SPLIT, 0, None, 0, None, st) == pent.OK
    pent.pent_sync()
    ref = oracle.batch_persys(*[host(t) for t in bands], F)
    assert max_rel_err(host(X), ref) < TOL_F32


def test_work_too_small_rejected():
    import torch
    N, batch = 16, 8
    bands = [torch.ones(N, batch, dtype=torch.float64, device="cuda") for _ in range(5)]
    X = torch.ones(N, batch, dtype=torch.float64, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        pent.pent_factor_solve(*bands, X, work=small)


def to_blocked(v, bs):
    """[N][batch] -> [batch / bs][N][bs]: the block-interleaved layout."""
    N, batch = v.shape
    return np.ascontiguousarray(v.reshape(N, batch // bs, bs).transpose(1, 0, 2))


def from_blocked(v):
    nb, N, bs = v.shape
    return v.transpose(1, 0, 2).reshape(N, nb * bs)


@pytest.mark.parametrize("variant,dtype,tol", [("split", np.float32, TOL_F32), ("thread", np.float32, TOL_F32),
                                               ("thread", np.float64, TOL_F64), ("thread_df", np.float64, TOL_F64)])
@pytest.mark.parametrize("bs", [8, 16, 48, 256])
@pytest.mark.parametrize("N", [17, 256, 300])
def test_block_interleaved(variant, dtype, tol, bs, N):
    """Blocks of bs systems, each an interleaved [N][bs] array (bs = 16, 48, 256: TMA boxes
    from 3-D tensor maps; bs = 8: per-thread cp.async), against the oracle."""
    batch = 768
    bands = inputs.persys_bands(N, batch, seed=N + bs, dtype=dtype)
    F = inputs.rhs_uniform(N, batch, seed=N + bs).astype(dtype)
    ref = oracle.batch_persys(*bands, F)
    dB = [dev(to_blocked(v, bs)) for v in bands]
    X = dev(to_blocked(F, bs))
    pent.pent_factor_solve(*dB, X, variant=variant, block_size=bs)
    pent.pent_sync()
    assert max_rel_err(from_blocked(host(X)), ref) < tol


def test_block_size_must_divide_batch():
    import torch
    bands = [torch.ones(2, 10, 8, dtype=torch.float32, device="cuda") for _ in range(5)]
    X = torch.ones(2, 10, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        pent.pent_factor_solve(*bands, X, block_size=16)      # shape says bs = 8
    L = pent.lib()
    import ctypes
    vp = [ctypes.c_void_p(t.data_ptr()) for t in bands]
    assert L.pent_factor_solve_ex(*vp, ctypes.c_void_p(X.data_ptr()), 10, 16, pent.F32, pent.VARIANT_AUTO,
                                  6, None, 0, None, None) == pent.ERR_INVALID_ARG


def test_fp64_quarter_size_sampled():
    """N=256, batch 65536, fp64 per-system bands (the double-float kernel, the fp64
    default): 1024 sampled systems against the oracle."""
    N, batch = 256, 65536
    a, b, c, d, e = inputs.persys_bands(N, batch, seed=2, dtype=np.float64)
    F = inputs.rhs_uniform(N, batch, seed=2)
    X, info, _ = run_gpu((a, b, c, d, e), F, np.float64)
    idx = inputs.sample_systems(batch, 1024)
    ref = oracle.batch_persys(a[:, idx], b[:, idx], c[:, idx], d[:, idx], e[:, idx], F[:, idx])
    assert max_rel_err(X[:, idx], ref) < TOL_F64
    assert np.all(info == 0)


def test_auto_takes_null_work_where_no_kernel_needs_it():
    """pent_factor_solve through the C ABI with work = NULL: accepted for fp32 systems
    of up to 512 rows (the partitioned kernel keeps every intermediate on chip),
    refused where the chosen kernel needs factor storage (fp64)."""
    import ctypes
    import torch
    L = pent.lib()
    N, batch = 256, 2048
    assert pent.pent_factor_solve_needs_work(N, batch, pent.F32) == 0
    assert pent.pent_factor_solve_needs_work(N, batch, pent.F64) == pent.pent_factor_solve_work_bytes(
        N, batch, pent.F64)
    bands = inputs.persys_bands(N, batch, seed=77, dtype=np.float32)
    F = inputs.rhs_uniform(N, batch, seed=78).astype(np.float32)
    A = [dev(b) for b in bands]
    X = dev(F)
    vp = [ctypes.c_void_p(t.data_ptr()) for t in A + [X]]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.pent_factor_solve(*vp, N, batch, pent.F32, None, 0, None, stream)
    assert st == pent.OK
    assert L.pent_sync(stream) == pent.OK
    assert max_rel_err(host(X), oracle.batch_persys(*bands, F)) < TOL_F32
    A64 = [dev(b.astype(np.float64)) for b in bands]
    X64 = dev(F.astype(np.float64))
    vp64 = [ctypes.c_void_p(t.data_ptr()) for t in A64 + [X64]]
    assert L.pent_factor_solve(*vp64, N, batch, pent.F64, None, 0, None, stream) == pent.ERR_INVALID_ARG

"""pent_factor_solve_noalloc, the per-system solve for callers that cannot allocate
device memory: it uses the library's fixed 16 MiB scratch array instead of a caller
buffer.  Called through the C ABI directly, against the CPU oracle and against
pent_factor_solve on the same inputs.

Cases: fp32 with N = 256 (the partitioned kernel, no scratch at all); fp32 with
N = 1024 and batch 2048, which needs exactly the 16 MiB of the static array (the
one-thread kernel's factor storage, 2 * N * batch * 4 bytes); fp64 with N = 300
(the double-float one-thread kernel, factor storage as float pairs).  Two calls in
a row per case, so the second call runs on whatever the first left in the shared
array.  One system more than the array holds is refused and leaves the data alone.

This file sorts last so that a run stopping at the first failure has run every
other test before it.
"""
import ctypes

import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F32, TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype,code,tol,N,batch",
                         [(np.float32, pent.F32, TOL_F32, 256, 8192),
                          (np.float32, pent.F32, TOL_F32, 1024, 2048),
                          (np.float64, pent.F64, TOL_F64, 300, 3000)])
def test_noalloc_matches_oracle_and_factor_solve_on_two_calls(dtype, code, tol, N, batch):
    import torch
    L = pent.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        seed = 100 * call + N
        bands_h = inputs.persys_bands(N, batch, seed=seed, dtype=dtype)
        F = inputs.rhs_uniform(N, batch, seed=seed).astype(dtype)
        bands = [dev(v) for v in bands_h]
        x_ref, x_new = dev(F), dev(F)
        info_ref = torch.full((batch,), -1, dtype=torch.int32, device="cuda")
        info_new = torch.full((batch,), -1, dtype=torch.int32, device="cuda")
        need = pent.pent_factor_solve_needs_work(N, batch, code)
        work = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        st = L.pent_factor_solve(*map(_vp, bands), _vp(x_ref), N, batch, code,
                                 _vp(work) if need else None, need, _vp(info_ref), stream)
        assert st == pent.OK
        st = L.pent_factor_solve_noalloc(*map(_vp, bands), _vp(x_new), N, batch, code,
                                         _vp(info_new), stream)
        assert st == pent.OK, pent.status_string(st)
        assert L.pent_sync(stream) == pent.OK
        xn = host(x_new)
        assert max_rel_err(xn, oracle.batch_persys(*bands_h, F)) < tol
        assert max_rel_err(xn, host(x_ref)) < tol
        assert np.array_equal(host(info_new), host(info_ref))
        assert np.all(host(info_new) == 0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    L = pent.lib()
    N, batch = 1024, 2049          # 2 * 1024 * 2049 * 4 bytes: one system more than 16 MiB
    t = torch.ones(N, batch, dtype=torch.float32, device="cuda")
    before = host(t).copy()
    st = L.pent_factor_solve_noalloc(*([_vp(t)] * 6), N, batch, pent.F32, None, None)
    assert st == pent.ERR_UNSUPPORTED
    assert np.array_equal(host(t), before)       # nothing was queued

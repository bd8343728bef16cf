"""The library's calls enqueue work only (no allocation, no synchronisation on the
common paths), so a step loop can be captured into a CUDA graph and replayed."""
import numpy as np
import pytest

import oracle
from implicit_pde_stepping_gb300 import inputs, pent
from tests.gpu_util import TOL_F64, dev, host, max_rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", ["auto", "split", "thread_df", "thread"])
def test_solve_captured_in_cuda_graph(variant):
    import torch
    N, batch = 512, 4096
    bands = inputs.hyper_bands(N, 1.0)
    plan = pent.pent_factor(bands, batch)
    if variant != "auto":
        plan.set_variant(variant)
    F1 = inputs.rhs_uniform(N, batch, seed=1)
    F2 = inputs.rhs_uniform(N, batch, seed=2)
    X = dev(F1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):          # warm-up outside the capture (kernel attributes)
        pent.pent_solve(plan, X, stream=s)
    s.synchronize()
    X.copy_(dev(F1))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pent.pent_solve(plan, X, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert max_rel_err(host(X), oracle.batch_shared(bands, F1)) < TOL_F64
    X.copy_(dev(F2))                     # replay on new data in the same buffer
    g.replay()
    torch.cuda.synchronize()
    assert max_rel_err(host(X), oracle.batch_shared(bands, F2)) < TOL_F64
    plan.close()


@pytest.mark.parametrize("kind", ["hyper", "ch", "cn"])
def test_time_steps_captured_in_cuda_graph(kind):
    import torch
    N, batch, steps = 512, 1024, 5
    sigma, k2 = (0.7, 0.2)
    plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
    C0 = inputs.ch_initial(N, batch) if kind == "ch" else inputs.rhs_uniform(N, batch, seed=3)
    C = dev(C0)
    s = torch.cuda.Stream()

    def call():
        if kind == "hyper":
            pent.hyperdiffusion_step(plan, C, steps, stream=s)
        elif kind == "ch":
            pent.ch_step(plan, C, k2, steps, stream=s)
        else:
            pent.cn_step(plan, C, steps, stream=s)

    with torch.cuda.stream(s):
        call()
    s.synchronize()
    C.copy_(dev(C0))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    g.replay()
    torch.cuda.synchronize()
    ref = {"hyper": lambda: oracle.batch_hyperdiffusion(C0, sigma, steps),
           "ch": lambda: oracle.batch_ch(C0, sigma, k2, steps),
           "cn": lambda: oracle.batch_cn(C0, sigma, steps)}[kind]()
    assert max_rel_err(host(C), ref) < TOL_F64
    plan.close()


@pytest.mark.parametrize("kind", ["persys", "tri"])
def test_per_system_solves_captured_in_cuda_graph(kind):
    """The partitioned fp32 kernels build their TMA tensor maps on the host at each
    call and pass them by value, so a captured call replays on whatever the captured
    buffers hold at replay time."""
    import torch
    from tests.gpu_util import TOL_F32
    N, batch = 256, 4096
    if kind == "persys":
        bands = [dev(v) for v in inputs.persys_bands(N, batch, seed=4)]
        ref = lambda F: oracle.batch_persys(*[host(b) for b in bands], F)  # noqa: E731
        call = lambda X, s: pent.pent_factor_solve(*bands, X, stream=s)  # noqa: E731
    else:
        bands = [dev(v) for v in inputs.tri_bands(N, batch, seed=4)]
        ref = lambda F: oracle.batch_tri(*[host(b) for b in bands], F)  # noqa: E731
        call = lambda X, s: pent.tri_factor_solve(*bands, X, stream=s)  # noqa: E731
    F1 = inputs.rhs_uniform(N, batch, seed=5).astype(np.float32)
    F2 = inputs.rhs_uniform(N, batch, seed=6).astype(np.float32)
    X = dev(F1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(X, s)
    s.synchronize()
    X.copy_(dev(F1))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(X, s)
    g.replay()
    torch.cuda.synchronize()
    assert max_rel_err(host(X), ref(F1)) < TOL_F32
    X.copy_(dev(F2))
    g.replay()
    torch.cuda.synchronize()
    assert max_rel_err(host(X), ref(F2)) < TOL_F32

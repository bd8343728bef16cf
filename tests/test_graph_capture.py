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

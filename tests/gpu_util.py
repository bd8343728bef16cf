"""Helpers for the GPU parity tests: device transfer and the error metric.

Metric: per system s, ||x_s - ref_s||_inf / ||ref_s||_inf (absolute when the
reference is zero), maximised over systems.  Tolerances: 1e-10 for one fp64
solve, 1e-8 after 2000 Cahn–Hilliard steps, 1e-4 for fp32 (against the fp64
oracle on the same fp32 inputs).
"""
import numpy as np

TOL_F64 = 1e-10
TOL_CH = 1e-8
TOL_F32 = 1e-4


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def max_rel_err(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(x - ref), axis=0)
    den = np.max(np.abs(ref), axis=0)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(num / den)) if num.size else 0.0


def random_dd_bands(N, rng, margin=1.0):
    """Random strictly diagonally dominant shared bands [5][N]."""
    b = rng.uniform(-1, 1, size=(5, N))
    for i in range(N):
        b[2, i] = margin + np.abs(b[[0, 1, 3, 4], i]).sum() + rng.uniform(0, 1)
    return b

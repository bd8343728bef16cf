"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no solver arithmetic: only a counter-based random generator
and the recipes of the five workloads.  Both the CUDA path and the CPU oracle
are fed from here, so parity never depends on how either side draws numbers.

Generator.  SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based hash:

    k1 = mix(seed ^ G)            G = 0x9E3779B97F4A7C15 (golden-ratio increment)
    k2 = mix(k1 ^ field)          field = a fixed tag per array (RHS, band a, ...)
    r  = mix(k2 + (idx + 1) * G)  idx = s * N + i  (system s, row i)
    u  = (r >> 11) * 2^-53        uniform on [0, 1)

mix(z) is the SplitMix64 finaliser.  Because the value of entry (i, s) depends
only on (seed, field, s, i), any subset of systems is generated identically
whatever the batch size.  Arrays come back interleaved, shape [N][batch]
(row i holds entry i of every system), the layout of the GPU path.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# field tags, one per independent array
F_RHS, F_A, F_B, F_C, F_D, F_E, F_DIAG, F_NORMAL1, F_NORMAL2, F_C0 = range(1, 11)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, field: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k1 = _mix(np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ _G], dtype=np.uint64))
        k2 = _mix(k1 ^ np.uint64(field))
    return k2[0]


def _uniform_flat(key: np.uint64, idx: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        r = _mix(key + (idx.astype(np.uint64) + np.uint64(1)) * _G)
    return (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform01(seed: int, field: int, N: int, systems) -> np.ndarray:
    """U[0,1) array, interleaved [N][len(systems)], entry (i, j) = u(seed, field, systems[j]*N + i)."""
    systems = np.asarray(systems, dtype=np.int64)
    key = _key(seed, field)
    out = np.empty((N, systems.shape[0]), dtype=np.float64)
    rows = np.arange(N, dtype=np.int64)

    def work(lo: int, hi: int) -> None:
        idx = systems[None, :] * np.int64(N) + rows[lo:hi, None]
        out[lo:hi] = _uniform_flat(key, idx)

    nthreads = max(1, min(16, os.cpu_count() or 1))
    step = max(1, -(-N // (4 * nthreads)))
    if N * systems.shape[0] < (1 << 20):
        work(0, N)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(lambda lo: work(lo, min(N, lo + step)), range(0, N, step)))
    return out


def uniform(seed, field, N, systems, lo, hi) -> np.ndarray:
    u = uniform01(seed, field, N, systems)
    u *= (hi - lo)
    u += lo
    return u


def _systems(batch, systems):
    return np.arange(batch, dtype=np.int64) if systems is None else np.asarray(systems, np.int64)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
def hyper_bands(N: int, sigma: float) -> np.ndarray:
    """Constant bands [sigma, -4 sigma, 1 + 6 sigma, -4 sigma, sigma] as a [5][N] array (a..e)."""
    v = np.array([sigma, -4.0 * sigma, 1.0 + 6.0 * sigma, -4.0 * sigma, sigma], dtype=np.float64)
    return np.repeat(v[:, None], N, axis=1)


def rhs_uniform(N: int, batch: int, seed: int = 0, systems=None, lo=-1.0, hi=1.0) -> np.ndarray:
    """Right-hand sides i.i.d. uniform[lo, hi], interleaved [N][batch] fp64."""
    return uniform(seed, F_RHS, N, _systems(batch, systems), lo, hi)


def fourier_modes(N: int, batch: int, kmax: int = 8, seed: int = 0, systems=None):
    """Per-system Fourier coefficients a_k, b_k ~ N(0,1), k = 1..kmax (Box–Muller).

    Returns (a, b) each [kmax][nsys]."""
    s = _systems(batch, systems)
    u1 = uniform01(seed, F_NORMAL1, 2 * kmax, s)
    u2 = uniform01(seed, F_NORMAL2, 2 * kmax, s)
    z = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)
    return z[:kmax], z[kmax:]


def fourier_initial(N: int, batch: int, kmax: int = 8, seed: int = 0, systems=None) -> np.ndarray:
    """C(x_j) = sum_k a_k cos(2 pi k x_j) + b_k sin(2 pi k x_j), x_j = j/N; interleaved [N][nsys]."""
    a, b = fourier_modes(N, batch, kmax, seed, systems)
    x = np.arange(N, dtype=np.float64) / N
    k = np.arange(1, kmax + 1, dtype=np.float64)
    ph = 2.0 * np.pi * k[:, None] * x[None, :]          # [kmax][N]
    return np.cos(ph).T @ a + np.sin(ph).T @ b             # [N][nsys]


def persys_bands(N: int, batch: int, seed: int = 0, systems=None, dtype=np.float32):
    """Strictly diagonally dominant per-system bands (a, b, c, d, e), interleaved [N][nsys].

    Off-diagonals i.i.d. uniform[-1, 1] (entries whose column is outside the
    matrix are set to zero), rounded to ``dtype``; diagonal = 1 + sum of |in-range
    off-diagonals of the row| + uniform[0, 1], rounded to ``dtype``.
    """
    s = _systems(batch, systems)
    offs = {}
    rows = np.arange(N)[:, None]
    for field, name, off in ((F_A, "a", -2), (F_B, "b", -1), (F_D, "d", 1), (F_E, "e", 2)):
        v = uniform(seed, field, N, s, -1.0, 1.0)
        col = rows[:, 0] + off
        v[(col < 0) | (col >= N), :] = 0.0
        offs[name] = v.astype(dtype)
    diag = 1.0 + uniform01(seed, F_DIAG, N, s)
    for name in ("a", "b", "d", "e"):
        diag += np.abs(offs[name].astype(np.float64))
    c = diag.astype(dtype)
    return offs["a"], offs["b"], c, offs["d"], offs["e"]


def tri_bands(N: int, batch: int, seed: int = 0, systems=None, dtype=np.float32):
    """Strictly diagonally dominant per-system tridiagonal bands (a, b, c), interleaved [N][nsys].

    a (column i-1) and c (column i+1) i.i.d. uniform[-1, 1], zero where the
    column is outside the matrix, rounded to ``dtype``; diagonal b = 1 + |a| + |c|
    + uniform[0, 1], rounded to ``dtype``.  The same draws as the lower and upper
    neighbours of ``persys_bands``, so the two generators share one recipe.
    """
    s = _systems(batch, systems)
    rows = np.arange(N)
    offs = []
    for field, off in ((F_B, -1), (F_D, 1)):
        v = uniform(seed, field, N, s, -1.0, 1.0)
        col = rows + off
        v[(col < 0) | (col >= N), :] = 0.0
        offs.append(v.astype(dtype))
    diag = 1.0 + uniform01(seed, F_DIAG, N, s)
    for v in offs:
        diag += np.abs(v.astype(np.float64))
    return offs[0], diag.astype(dtype), offs[1]


def ch_initial(N: int, batch: int, seed: int = 0, systems=None) -> np.ndarray:
    """Cahn–Hilliard initial data C^0 i.i.d. uniform[-0.1, 0.1], interleaved [N][nsys]."""
    return uniform(seed, F_C0, N, _systems(batch, systems), -0.1, 0.1)


def sample_systems(batch: int, count: int) -> np.ndarray:
    """Deterministic, evenly spread subset of system indices (always includes 0 and batch-1)."""
    count = max(1, min(batch, count))
    if count == 1:
        return np.array([0], dtype=np.int64)
    return np.unique(np.round(np.linspace(0, batch - 1, count)).astype(np.int64))


def ch_params(N: int, gamma: float = 1e-4, dt_factor: float = 0.1):
    """(sigma, dt/dx^2) of the semi-implicit Cahn–Hilliard workload on [0, 1), dx = 1/N,
    dt = dt_factor dx^2:  sigma = gamma dt / dx^4, dt/dx^2 = dt_factor."""
    dx = 1.0 / N
    dt = dt_factor * dx * dx
    return gamma * dt / dx ** 4, dt / (dx * dx)


__all__ = [
    "uniform01", "uniform", "hyper_bands", "rhs_uniform", "fourier_modes", "fourier_initial",
    "persys_bands", "ch_initial", "sample_systems", "ch_params",
]

"""CPU reference oracle for the batched pentadiagonal solves — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it never imports the CUDA library: the two share no code.

The arithmetic lives in ``pent_oracle.c`` (plain C, fp64, one system per row as
in the serial validation code of "cuPentBatch – A batched pentadiagonal solver
for NVIDIA GPUs").  This module only compiles it with gcc, loads it with ctypes
and converts between the interleaved layout ``[N][batch]`` (row i holds entry i
of every system) and the one-system-per-row layout the C code uses.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pent_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ZERO_PIVOT, ENOMEM = 0, 1, 2, 3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``pent_oracle.c`` into ``liboracle.so`` (OpenMP if gcc supports it).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so the
    oracle gives the same bits on x86-64 and AArch64.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        r = subprocess.run(base + extra + [_SRC, "-o", tmp, "-lm"], capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB)
            return _LIB
    raise OracleError("gcc failed to build the oracle:\n" + r.stderr)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_num_threads.restype = i
            lib.oracle_pent_factor.argtypes = [i] + [dp] * 10
            lib.oracle_pent_solve.argtypes = [i] + [dp] * 7
            lib.oracle_cyclic_solve.argtypes = [i] + [dp] * 7
            lib.oracle_batch_shared.argtypes = [i, i, dp, i, dp, dp]
            lib.oracle_batch_persys.argtypes = [i, i] + [dp] * 7
            lib.oracle_batch_hyperdiffusion.argtypes = [i, i, d, i, dp]
            lib.oracle_batch_ch.argtypes = [i, i, d, d, i, dp]
            lib.oracle_batch_cn.argtypes = [i, i, d, i, dp]
            lib.oracle_tri_solve.argtypes = [i, dp, dp, dp, dp, dp]
            lib.oracle_batch_tri.argtypes = [i, i, dp, dp, dp, dp, dp]
            for fn in ("oracle_pent_factor", "oracle_pent_solve", "oracle_cyclic_solve",
                       "oracle_batch_shared", "oracle_batch_persys",
                       "oracle_batch_hyperdiffusion", "oracle_batch_ch", "oracle_batch_cn",
                       "oracle_tri_solve", "oracle_batch_tri"):
                getattr(lib, fn).restype = i
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise OracleError(f"{what}: oracle returned code {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------------------
# single-system entry points (vectors of length N)
# ----------------------------------------------------------------------------
def factor(a, b, c, d, e):
    """LR factorisation (factorisation steps 1–14): returns alpha, beta, gamma, delta, eps."""
    a, b, c, d, e = (_f64(v) for v in (a, b, c, d, e))
    N = c.shape[0]
    out = [np.empty(N) for _ in range(5)]
    _check(_load().oracle_pent_factor(N, _p(a), _p(b), _p(c), _p(d), _p(e), *map(_p, out)),
           "factor")
    return tuple(out)


def solve(a, b, c, d, e, f, cyclic: bool = False) -> np.ndarray:
    """Solve one pentadiagonal system (non-cyclic LR or cyclic bordering)."""
    a, b, c, d, e, f = (_f64(v) for v in (a, b, c, d, e, f))
    N = c.shape[0]
    x = np.empty(N)
    fn = _load().oracle_cyclic_solve if cyclic else _load().oracle_pent_solve
    _check(fn(N, _p(a), _p(b), _p(c), _p(d), _p(e), _p(f), _p(x)), "solve")
    return x


# ----------------------------------------------------------------------------
# batched entry points, interleaved arrays [N][batch]
# ----------------------------------------------------------------------------
def _rows(x_il: np.ndarray) -> np.ndarray:
    """interleaved [N][batch] -> one system per row [batch][N] (always a fresh fp64 copy)."""
    return np.array(np.asarray(x_il, dtype=np.float64).T, dtype=np.float64, order="C", copy=True)


def batch_shared(bands, F_il, cyclic: bool = False) -> np.ndarray:
    """Shared-matrix batch solve.  bands: [5][N] (a, b, c, d, e); F_il: [N][batch]."""
    bands = _f64(bands)
    N = bands.shape[1]
    X = _rows(F_il)
    batch = X.shape[0]
    _check(_load().oracle_batch_shared(N, batch, _p(bands), int(bool(cyclic)), _p(X), _p(X)),
           "batch_shared")
    return np.ascontiguousarray(X.T)


def batch_persys(A_il, B_il, C_il, D_il, E_il, F_il) -> np.ndarray:
    """Per-system batch solve; every array interleaved [N][batch] (widened to fp64)."""
    A, B, C, D, E = (_rows(v) for v in (A_il, B_il, C_il, D_il, E_il))
    X = _rows(F_il)
    batch, N = X.shape
    _check(_load().oracle_batch_persys(N, batch, _p(A), _p(B), _p(C), _p(D), _p(E), _p(X), _p(X)),
           "batch_persys")
    return np.ascontiguousarray(X.T)


def batch_hyperdiffusion(C_il, sigma: float, nsteps: int) -> np.ndarray:
    """nsteps of C <- (I + sigma D4)^{-1} C, periodic, on interleaved [N][batch]."""
    X = _rows(C_il)
    batch, N = X.shape
    _check(_load().oracle_batch_hyperdiffusion(N, batch, float(sigma), int(nsteps), _p(X)),
           "batch_hyperdiffusion")
    return np.ascontiguousarray(X.T)


def batch_ch(C_il, sigma: float, dt_over_dx2: float, nsteps: int) -> np.ndarray:
    """nsteps of semi-implicit Cahn–Hilliard on interleaved [N][batch]."""
    X = _rows(C_il)
    batch, N = X.shape
    _check(_load().oracle_batch_ch(N, batch, float(sigma), float(dt_over_dx2), int(nsteps), _p(X)),
           "batch_ch")
    return np.ascontiguousarray(X.T)


def batch_cn(C_il, sigma_x: float, nsteps: int) -> np.ndarray:
    """nsteps of Crank–Nicolson hyperdiffusion (I + sx D4) C' = (I - sx D4) C, periodic."""
    X = _rows(C_il)
    batch, N = X.shape
    _check(_load().oracle_batch_cn(N, batch, float(sigma_x), int(nsteps), _p(X)), "batch_cn")
    return np.ascontiguousarray(X.T)


def tri_solve(a, b, c, y) -> np.ndarray:
    """One tridiagonal system by the Thomas algorithm (fp64)."""
    a, b, c, y = (np.ascontiguousarray(v, dtype=np.float64) for v in (a, b, c, y))
    u = np.empty_like(y)
    _check(_load().oracle_tri_solve(len(y), _p(a), _p(b), _p(c), _p(y), _p(u)), "tri_solve")
    return u


def batch_tri(A_il, B_il, C_il, Y_il) -> np.ndarray:
    """Per-system tridiagonal batch; every array interleaved [N][batch] (widened to fp64)."""
    A, B, C = (_rows(v) for v in (A_il, B_il, C_il))
    Y = _rows(Y_il)
    batch, N = Y.shape
    U = np.empty_like(Y)
    _check(_load().oracle_batch_tri(N, batch, _p(A), _p(B), _p(C), _p(Y), _p(U)), "batch_tri")
    return np.ascontiguousarray(U.T)


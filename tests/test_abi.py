"""The C-ABI library loads and exports every symbol include/pent.h declares; host-side
argument checks reject bad calls before anything reaches the GPU.  No GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest

from implicit_pde_stepping_gb300 import build, pent

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def L():
    build.build()
    return pent.lib()


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "for", "while", "sizeof"):
                names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_api():
    names = declared_functions()
    for fn in ("pent_factor", "pent_solve", "pent_factor_solve", "hyperdiffusion_step", "ch_step",
               "cn_step", "pent_destroy", "pent_status_string", "pent_sync"):
        assert fn in names


def test_every_declared_symbol_is_exported(L):
    for fn in declared_functions():
        assert hasattr(L, fn), f"{fn} declared in include/*.h but not exported by libpent.so"


def test_status_strings(L):
    assert pent.status_string(pent.OK) == "PENT_OK"
    assert pent.status_string(pent.ERR_ZERO_PIVOT) == "PENT_ERR_ZERO_PIVOT"
    assert pent.status_string(99) == "PENT_ERR_UNKNOWN"


def test_argument_errors_before_any_device_work(L):
    h = ctypes.c_void_p()
    bands = np.ones((5, 8))
    bp = bands.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    assert L.pent_factor(bp, 0, 1, 0, 0, ctypes.byref(h)) == pent.ERR_INVALID_ARG
    assert L.pent_factor(bp, 4, 1, 1, 0, ctypes.byref(h)) == pent.ERR_INVALID_ARG  # cyclic N < 5
    assert L.pent_factor(bp, 8, 0, 0, 0, ctypes.byref(h)) == pent.ERR_INVALID_ARG  # batch 0
    assert L.pent_factor(bp, 8, 1, 2, 0, ctypes.byref(h)) == pent.ERR_INVALID_ARG  # cyclic flag
    assert L.pent_factor(bp, 8, 1, 0, 7, ctypes.byref(h)) == pent.ERR_INVALID_ARG  # dtype
    assert L.pent_factor(None, 8, 1, 0, 0, ctypes.byref(h)) == pent.ERR_INVALID_ARG
    assert h.value is None
    assert L.pent_solve(None, ctypes.c_void_p(256), 1, None) == pent.ERR_INVALID_ARG
    assert L.hyperdiffusion_step(None, ctypes.c_void_p(256), 1, 1, None) == pent.ERR_INVALID_ARG
    assert L.ch_step(None, ctypes.c_void_p(256), 1, 0.1, 1, None) == pent.ERR_INVALID_ARG
    assert L.cn_step(None, ctypes.c_void_p(256), 1, 1, None) == pent.ERR_INVALID_ARG
    z = ctypes.c_void_p(0)
    assert L.pent_factor_solve(z, z, z, z, z, z, 8, 1, 0, z, 0, z, z) == pent.ERR_INVALID_ARG
    assert L.pent_set_variant(None, 0) == pent.ERR_INVALID_ARG
    L.pent_destroy(None)


def test_work_bytes(L):
    assert pent.pent_factor_solve_work_bytes(256, 262144, pent.F32) == 2 * 256 * 262144 * 4
    assert pent.pent_factor_solve_work_bytes(10, 3, pent.F64) == 2 * 10 * 3 * 8
    assert L.pent_factor_solve_work_bytes(0, 3, 0) == 0


def test_launch_counter_starts_readable(L):
    assert pent.launch_count() >= 0


def test_per_system_argument_errors_before_any_device_work(L):
    """The per-system entry points reject bad arguments on the host: null or
    misaligned pointers, sizes, a block size that does not divide the batch, an
    unknown dtype, and variants that do not exist for the dtype or size."""
    ok = ctypes.c_void_p(1 << 12)            # aligned, never dereferenced on these paths
    mis = ctypes.c_void_p((1 << 12) + 8)     # 8-byte aligned only
    z = ctypes.c_void_p(0)
    work = ctypes.c_void_p(1 << 16)
    p6 = [ok] * 6
    ex = L.pent_factor_solve_ex
    assert ex(*p6, 0, 4, pent.F64, pent.VARIANT_AUTO, 0, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert ex(*p6, 8, 0, pent.F64, pent.VARIANT_AUTO, 0, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert ex(z, *p6[1:], 8, 4, pent.F64, pent.VARIANT_AUTO, 0, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert ex(*p6[:5], mis, 8, 4, pent.F64, pent.VARIANT_AUTO, 0, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert ex(*p6, 8, 6, pent.F64, pent.VARIANT_AUTO, 4, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert ex(*p6, 8, 4, 7, pent.VARIANT_AUTO, 0, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    # the double-float kernel is for fp64 systems; the partitioned one for fp32, N <= 512
    assert ex(*p6, 8, 4, pent.F32, pent.VARIANT_THREAD_DF, 0, work, 1 << 20, None, None) == pent.ERR_UNSUPPORTED
    assert ex(*p6, 8, 4, pent.F64, pent.VARIANT_SPLIT, 0, work, 1 << 20, None, None) == pent.ERR_UNSUPPORTED
    assert ex(*p6, 600, 4, pent.F32, pent.VARIANT_SPLIT, 0, work, 1 << 20, None, None) == pent.ERR_UNSUPPORTED
    tri = L.tri_factor_solve
    p4 = [ok] * 4
    assert tri(z, *p4[1:], 8, 4, pent.F64, pent.VARIANT_AUTO, 0, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert tri(*p4, 8, 6, pent.F32, pent.VARIANT_AUTO, 4, work, 1 << 20, None, None) == pent.ERR_INVALID_ARG
    assert tri(*p4, 8, 4, pent.F32, pent.VARIANT_THREAD_DF, 0, work, 1 << 20, None, None) == pent.ERR_UNSUPPORTED
    assert tri(*p4, 8, 4, pent.F64, pent.VARIANT_SPLIT, 0, work, 1 << 20, None, None) == pent.ERR_UNSUPPORTED
    na = L.pent_factor_solve_noalloc
    assert na(*p6, 0, 4, pent.F32, None, None) == pent.ERR_INVALID_ARG
    assert na(*p6[:5], mis, 8, 4, pent.F32, None, None) == pent.ERR_INVALID_ARG
    assert na(*p6, 8, 4, 9, None, None) == pent.ERR_INVALID_ARG
    assert L.pent_solve_host(None, ok, ok, 4, 0, None) == pent.ERR_INVALID_ARG
    assert L.pent_get_variant(None, 4) == pent.VARIANT_AUTO


def test_factor_solve_needs_work():
    """The AUTO per-system solve needs no scratch where the fp32 partitioned kernel runs
    (N <= 512) and the one-thread kernels' factor storage elsewhere."""
    L = pent.lib()
    assert pent.pent_factor_solve_needs_work(256, 262144, pent.F32) == 0
    assert pent.pent_factor_solve_needs_work(512, 7, pent.F32) == 0
    assert pent.pent_factor_solve_needs_work(513, 7, pent.F32) == 2 * 513 * 7 * 4
    assert pent.pent_factor_solve_needs_work(256, 3, pent.F64) == 2 * 256 * 3 * 8
    assert L.pent_factor_solve_needs_work(0, 3, 0) == 0
    assert L.pent_factor_solve_needs_work(3, 3, 7) == 0

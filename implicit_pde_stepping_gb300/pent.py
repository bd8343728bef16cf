"""Python binding of libpent (the C ABI in include/pent.h), via ctypes.

Argument marshalling only: every solve runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  The binding refuses to work if
``libpent.so`` has not been built; there is no fallback of any kind.

Arrays are torch tensors on the current CUDA device in the interleaved layout
``[N][batch]`` (row i holds entry i of every system), contiguous.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpent.so")

OK, ERR_INVALID_ARG, ERR_ZERO_PIVOT, ERR_CUDA, ERR_ALLOC, ERR_UNSUPPORTED = range(6)
F64, F32 = 0, 1
VARIANT_AUTO, VARIANT_THREAD, VARIANT_THREAD_DF, VARIANT_SPLIT = range(4)
VARIANTS = {"auto": VARIANT_AUTO, "thread": VARIANT_THREAD, "thread_df": VARIANT_THREAD_DF,
            "split": VARIANT_SPLIT}
# plan options (pent_set_option; tuning and testing hooks, see include/pent.h)
OPTIONS = {"fixed_grid": 1, "serial_chunk_scan": 2, "border_all_chunks": 3, "multi_step": 4,
           "cheap_terms": 5, "chunk_dedup": 6, "twisted_ring": 7, "steps_systems": 8,
           "twisted_systems_per_cta": 9, "twisted_systems_per_thread": 10,
           "twisted_prefetch_rows": 11, "persistent_ctas": 12}

_lock = threading.Lock()
_lib = None


class PentError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def lib():
    """Load libpent.so (built by implicit_pde_stepping_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libpent.so is not built ({LIB_PATH}); run "
                                   "`python -m implicit_pde_stepping_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, d, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
            L.pent_factor.argtypes = [ctypes.POINTER(ctypes.c_double), i, i, i, i,
                                      ctypes.POINTER(vp)]
            L.pent_solve.argtypes = [vp, vp, i, vp]
            L.pent_solve_host.argtypes = [vp, vp, vp, i, i, vp]
            L.pent_factor_solve.argtypes = [vp] * 6 + [i, i, i, vp, sz, vp, vp]
            L.pent_factor_solve_ex.argtypes = [vp] * 6 + [i, i, i, i, i, vp, sz, vp, vp]
            L.pent_factor_solve_work_bytes.argtypes = [i, i, i]
            L.pent_factor_solve_work_bytes.restype = sz
            L.pent_factor_solve_needs_work.argtypes = [i, i, i]
            L.pent_factor_solve_needs_work.restype = sz
            L.pent_factor_solve_noalloc.argtypes = [vp] * 6 + [i, i, i, vp, vp]
            L.pent_factor_solve_noalloc.restype = i
            L.hyperdiffusion_step.argtypes = [vp, vp, i, i, vp]
            L.ch_step.argtypes = [vp, vp, i, d, i, vp]
            L.cn_step.argtypes = [vp, vp, i, i, vp]
            L.tri_factor_solve_work_bytes.argtypes = [i, i, i]
            L.tri_factor_solve_work_bytes.restype = sz
            L.tri_factor_solve.argtypes = [vp] * 4 + [i, i, i, i, i, vp, sz, vp, vp]
            L.pent_set_variant.argtypes = [vp, i]
            L.pent_get_variant.argtypes = [vp, i]
            L.pent_set_option.argtypes = [vp, i, i]
            L.pent_plan_error.argtypes = [vp]
            L.pent_destroy.argtypes = [vp]
            L.pent_destroy.restype = None
            L.pent_sync.argtypes = [vp]
            L.pent_status_string.argtypes = [i]
            L.pent_status_string.restype = ctypes.c_char_p
            L.pent_launch_count.argtypes = []
            L.pent_launch_count.restype = ctypes.c_ulonglong
            for fn in ("pent_factor", "pent_solve", "pent_solve_host", "pent_factor_solve",
                       "pent_factor_solve_ex",
                       "hyperdiffusion_step",
                       "ch_step", "cn_step", "tri_factor_solve", "pent_set_variant", "pent_set_option", "pent_plan_error",
                       "pent_get_variant", "pent_sync"):
                getattr(L, fn).restype = i
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pent_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise PentError(status, what)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float64:
        return F64
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t, N=None, dtype=None, what="array"):
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.dim() != 2:
        raise ValueError(f"{what} must be [N][batch]")
    if N is not None and t.shape[0] != N:
        raise ValueError(f"{what} has {t.shape[0]} rows, expected {N}")
    if dtype is not None and _dtype_code(t) != dtype:
        raise TypeError(f"{what} dtype does not match")
    return ctypes.c_void_p(t.data_ptr())


class Plan:
    """A factored shared matrix (owns the device tables; freed on close/GC)."""

    def __init__(self, handle, N, batch, cyclic, dtype):
        self._h = handle
        self.N, self.batch, self.cyclic, self.dtype = N, batch, cyclic, dtype

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("plan is closed")
        return self._h

    def close(self):
        if self._h is not None:
            lib().pent_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_variant(self, variant):
        code = VARIANTS[variant] if isinstance(variant, str) else int(variant)
        _check(lib().pent_set_variant(self.handle, code), "pent_set_variant")

    def set_option(self, option, value: int):
        """pent_set_option: a tuning / testing hook (names in OPTIONS)."""
        code = OPTIONS[option] if isinstance(option, str) else int(option)
        _check(lib().pent_set_option(self.handle, code, int(value)), "pent_set_option")

    def error(self) -> int:
        """pent_plan_error: PENT_ERR_CUDA if a kernel of this plan gave up waiting for a copy."""
        return int(lib().pent_plan_error(self.handle))

    def variant(self, batch=None) -> int:
        return int(lib().pent_get_variant(self.handle, int(batch or self.batch)))


def pent_factor(bands, batch: int, cyclic: bool = False, dtype: str = "f64") -> Plan:
    """Factor a shared matrix.  bands: [5][N] array-like (a, b, c, d, e) on the host."""
    b = np.ascontiguousarray(np.asarray(bands, dtype=np.float64))
    if b.ndim != 2 or b.shape[0] != 5:
        raise ValueError("bands must be [5][N]")
    N = b.shape[1]
    code = F64 if dtype in ("f64", "float64", F64) else F32
    h = ctypes.c_void_p()
    _check(lib().pent_factor(b.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), N, int(batch),
                             int(bool(cyclic)), code, ctypes.byref(h)), "pent_factor")
    return Plan(h, N, int(batch), bool(cyclic), code)


def pent_solve(plan: Plan, rhs, stream=None) -> None:
    """In-place shared-matrix solve of rhs ([N][batch] CUDA tensor)."""
    p = _ptr(rhs, plan.N, plan.dtype, "rhs")
    _check(lib().pent_solve(plan.handle, p, int(rhs.shape[1]), _stream(stream)), "pent_solve")


def pent_solve_host(plan: Plan, rhs_host, x_host=None, chunks: int = 0, stream=None):
    """Shared-matrix solve of a HOST tensor ([N][batch], pinned for asynchronous copies):
    copy in, solve and copy out overlapped in blocks of systems.  Returns x_host (a new
    pinned tensor if None); valid once the stream reaches this call (e.g. pent_sync)."""
    import torch
    if rhs_host.is_cuda or (x_host is not None and x_host.is_cuda):
        raise ValueError("pent_solve_host takes host tensors")
    if rhs_host.dim() != 2 or rhs_host.shape[0] != plan.N or not rhs_host.is_contiguous():
        raise ValueError("rhs_host must be a contiguous [N][batch] host tensor")
    if _dtype_code(rhs_host) != plan.dtype:
        raise TypeError("rhs_host dtype does not match the plan")
    if x_host is None:
        x_host = torch.empty_like(rhs_host).pin_memory()
    if x_host.shape != rhs_host.shape or x_host.dtype != rhs_host.dtype or not x_host.is_contiguous():
        raise ValueError("x_host must match rhs_host")
    _check(lib().pent_solve_host(plan.handle, ctypes.c_void_p(rhs_host.data_ptr()),
                                 ctypes.c_void_p(x_host.data_ptr()), int(rhs_host.shape[1]), int(chunks),
                                 _stream(stream)), "pent_solve_host")
    return x_host


def pent_factor_solve_work_bytes(N: int, batch: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (F64 if str(dtype).endswith("64") else F32)
    return int(lib().pent_factor_solve_work_bytes(int(N), int(batch), code))


def pent_factor_solve_needs_work(N: int, batch: int, dtype) -> int:
    """Scratch bytes the AUTO variant needs (0 where the partitioned kernel runs)."""
    code = dtype if isinstance(dtype, int) else (F64 if str(dtype).endswith("64") else F32)
    return int(lib().pent_factor_solve_needs_work(int(N), int(batch), code))


def pent_factor_solve(a, b, c, d, e, rhs, work=None, info=None, stream=None, variant: str = "auto",
                      block_size: int = 0):
    """Per-system factor + solve, in place in rhs.  variant: "auto", "thread" or "split"
    (fp32, N <= 512).  work: a CUDA uint8 tensor of at least pent_factor_solve_work_bytes()
    bytes (allocated here if None; unused by the split kernel).  info: CUDA int32 [batch].
    block_size 0: arrays interleaved [N][batch]; block_size bs > 0: block-interleaved,
    arrays shaped [batch / bs][N][bs]."""
    import torch
    if block_size:
        nb, N, bs = rhs.shape
        if bs != block_size:
            raise ValueError("block-interleaved arrays must be [batch / bs][N][bs]")
        batch = nb * bs
        for t, n in zip((a, b, c, d, e, rhs), "abcder"):
            if t.shape != rhs.shape or not t.is_cuda or not t.is_contiguous() or t.dtype != rhs.dtype:
                raise ValueError(f"{n} must match rhs: contiguous CUDA [batch / bs][N][bs]")
        code = _dtype_code(rhs)
        ptrs = [ctypes.c_void_p(t.data_ptr()) for t in (a, b, c, d, e)]
        rp = ctypes.c_void_p(rhs.data_ptr())
    else:
        N, batch = rhs.shape
        code = _dtype_code(rhs)
        ptrs = [_ptr(t, N, code, n) for t, n in zip((a, b, c, d, e), "abcde")]
        rp = _ptr(rhs, N, code, "rhs")
    # scratch only where the chosen kernel uses it (none for the fp32 partitioned kernel)
    need = (pent_factor_solve_needs_work(N, batch, code) if variant == "auto" and not block_size
            else pent_factor_solve_work_bytes(N, batch, code))
    if variant == "split":
        need = 0
    if work is None and need > 0:
        work = torch.empty(need, dtype=torch.uint8, device=rhs.device)
    nbytes = 0 if work is None else work.numel() * work.element_size()
    if nbytes < need:
        raise ValueError("work too small")
    ip = None
    if info is not None:
        if info.dtype != torch.int32 or info.numel() < batch or not info.is_cuda:
            raise ValueError("info must be a CUDA int32 tensor of >= batch elements")
        ip = ctypes.c_void_p(info.data_ptr())
    wp = ctypes.c_void_p(work.data_ptr() if work is not None else None)
    _check(lib().pent_factor_solve_ex(*ptrs, rp, N, batch, code, VARIANTS[variant], int(block_size),
                                      wp, nbytes, ip, _stream(stream)), "pent_factor_solve")
    return work


def pent_factor_solve_noalloc(a, b, c, d, e, rhs, info=None, stream=None) -> None:
    """Per-system factor + solve in place, with the library's fixed 16 MiB scratch instead of
    caller memory (for callers that cannot allocate device memory; see include/pent.h)."""
    import torch
    N, batch = rhs.shape
    code = _dtype_code(rhs)
    ptrs = [_ptr(t, N, code, n) for t, n in zip((a, b, c, d, e), "abcde")]
    ip = None
    if info is not None:
        if info.dtype != torch.int32 or info.numel() < batch or not info.is_cuda:
            raise ValueError("info must be a CUDA int32 tensor of >= batch elements")
        ip = ctypes.c_void_p(info.data_ptr())
    _check(lib().pent_factor_solve_noalloc(*ptrs, _ptr(rhs, N, code, "rhs"), N, batch, code, ip,
                                           _stream(stream)), "pent_factor_solve_noalloc")


def tri_factor_solve_work_bytes(N: int, batch: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (F64 if str(dtype).endswith("64") else F32)
    return int(lib().tri_factor_solve_work_bytes(int(N), int(batch), code))


def tri_factor_solve(a, b, c, rhs, variant: str = "auto", work=None, info=None, stream=None,
                     block_size: int = 0):
    """Per-system tridiagonal solve in place in rhs (Thomas algorithm).  variant: "auto",
    "thread" or "split".  work: CUDA uint8 tensor of tri_factor_solve_work_bytes() bytes
    (allocated here if None; unused by the split kernel).  info: CUDA int32 [batch].
    block_size 0: arrays interleaved [N][batch]; block_size bs > 0: block-interleaved,
    arrays shaped [batch / bs][N][bs]."""
    import torch
    if block_size:
        nb, N, bs = rhs.shape
        if bs != block_size:
            raise ValueError("block-interleaved arrays must be [batch / bs][N][bs]")
        batch = nb * bs
        for t, n in zip((a, b, c, rhs), "abcr"):
            if t.shape != rhs.shape or not t.is_cuda or not t.is_contiguous() or t.dtype != rhs.dtype:
                raise ValueError(f"{n} must match rhs: contiguous CUDA [batch / bs][N][bs]")
        code = _dtype_code(rhs)
        ptrs = [ctypes.c_void_p(t.data_ptr()) for t in (a, b, c)]
        rp = ctypes.c_void_p(rhs.data_ptr())
    else:
        N, batch = rhs.shape
        code = _dtype_code(rhs)
        ptrs = [_ptr(t, N, code, n) for t, n in zip((a, b, c), "abc")]
        rp = _ptr(rhs, N, code, "rhs")
    # scratch only where the chosen kernel uses it (none for the fp32 partitioned kernel)
    split_runs = code == F32 and N <= 512 and variant in ("auto", "split")
    need = 0 if split_runs else tri_factor_solve_work_bytes(N, batch, code)
    if work is None and need > 0:
        work = torch.empty(need, dtype=torch.uint8, device=rhs.device)
    nbytes = 0 if work is None else work.numel() * work.element_size()
    ip = None
    if info is not None:
        if info.dtype != torch.int32 or info.numel() < batch or not info.is_cuda:
            raise ValueError("info must be a CUDA int32 tensor of >= batch elements")
        ip = ctypes.c_void_p(info.data_ptr())
    wp = ctypes.c_void_p(work.data_ptr() if work is not None else None)
    _check(lib().tri_factor_solve(*ptrs, rp, N, batch, code, VARIANTS[variant], int(block_size),
                                  wp, nbytes, ip, _stream(stream)), "tri_factor_solve")
    return work


def hyperdiffusion_step(plan: Plan, C, nsteps: int, stream=None) -> None:
    p = _ptr(C, plan.N, plan.dtype, "C")
    _check(lib().hyperdiffusion_step(plan.handle, p, int(C.shape[1]), int(nsteps), _stream(stream)),
           "hyperdiffusion_step")


def ch_step(plan: Plan, C, dt_over_dx2: float, nsteps: int, stream=None) -> None:
    p = _ptr(C, plan.N, plan.dtype, "C")
    _check(lib().ch_step(plan.handle, p, int(C.shape[1]), float(dt_over_dx2), int(nsteps),
                         _stream(stream)), "ch_step")


def cn_step(plan: Plan, C, nsteps: int, stream=None) -> None:
    """nsteps of Crank–Nicolson: C <- A^{-1} (2I - A) C for the plan's cyclic A."""
    p = _ptr(C, plan.N, plan.dtype, "C")
    _check(lib().cn_step(plan.handle, p, int(C.shape[1]), int(nsteps), _stream(stream)), "cn_step")


def pent_sync(stream=None) -> None:
    _check(lib().pent_sync(_stream(stream)), "pent_sync")


def launch_count() -> int:
    return int(lib().pent_launch_count())

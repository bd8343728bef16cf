"""The oracle pins are sensitive: each plausible mistake planted in a copy of the
oracle (a dropped term, a flipped sign, a wrong index, a transposed operand) makes
at least one pin of test_oracle.py fail.  CPU only; the planted copy is built in
a temporary directory and never replaces the real oracle."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from tests import test_oracle as T

SRC = os.path.join(os.path.dirname(oracle.__file__), "pent_oracle.c")

MUTATIONS = [
    ("beta sign", "beta[i] = bi - ai * gm2;", "beta[i] = bi + ai * gm2;"),
    ("alpha dropped term", "alpha[i] = ci - ai * dm2 - beta[i] * gm1;", "alpha[i] = ci - beta[i] * gm1;"),
    ("gamma wrong operand", "gamma[i] = (di - beta[i] * dm1) / alpha[i];",
     "gamma[i] = (di - beta[i] * gm1) / alpha[i];"),
    ("delta multiply", "delta[i] = ei / alpha[i];", "delta[i] = ei * alpha[i];"),
    ("forward wrong index", "g[i] = (f[i] - eps[i] * gm2 - beta[i] * gm1) / alpha[i];",
     "g[i] = (f[i] - eps[i] * gm1 - beta[i] * gm1) / alpha[i];"),
    ("backward wrong index", "x[i] = g[i] - gamma[i] * xp1 - delta[i] * xp2;",
     "x[i] = g[i] - gamma[i] * xp1 - delta[i] * xp1;"),
    ("alpha wrong index", "alpha[i] = ci - ai * dm2 - beta[i] * gm1;",
     "alpha[i] = ci - ai * dm2 - beta[i] * gm2;"),
    ("schur transposed", "S01 -= H0[j] * Y1[j];", "S01 -= H1[j] * Y0[j];"),
    ("cramer operand", "double xt0 = (r0 * S11 - S01 * r1) / det;",
     "double xt0 = (r0 * S11 - S10 * r1) / det;"),
    ("tail swap", "x[j] = Yf[j] - Y0[j] * xt0 - Y1[j] * xt1;",
     "x[j] = Yf[j] - Y0[j] * xt1 - Y1[j] * xt0;"),
    ("border columns swapped", "if (col == M) G0[i] += v; else G1[i] += v;",
     "if (col == M) G1[i] += v; else G0[i] += v;"),
    ("D2 sign", "rhs[i] = C[i] + dt_over_dx2 * (u[im] - 2.0 * u[i] + u[ip]);",
     "rhs[i] = C[i] + dt_over_dx2 * (u[im] - 2.0 * u[i] - u[ip]);"),
    ("cubic sign", "u[i] = C[i] * C[i] * C[i] - C[i];", "u[i] = C[i] * C[i] * C[i] + C[i];"),
    ("cubic power", "u[i] = C[i] * C[i] * C[i] - C[i];", "u[i] = C[i] * C[i] - C[i];"),
    ("D4 band sign", "b[i] = -4.0 * sigma;", "b[i] = 4.0 * sigma;"),
    ("CN explicit half sign", "rhs[i] = C[i] - sigma_x * d4;", "rhs[i] = C[i] + sigma_x * d4;"),
    ("CN stencil index", "double d4 = C[im2] - 4.0 * C[im1] + 6.0 * C[i] - 4.0 * C[ip1] + C[ip2];",
     "double d4 = C[im2] - 4.0 * C[im1] + 6.0 * C[i] - 4.0 * C[ip1] + C[ip1];"),
    ("CN wrap", "int im2 = (i + N - 2) % N,", "int im2 = (i + N - 1) % N,"),
    ("Thomas denominator sign", "const double den = b[i] - cprev * ai;",
     "const double den = b[i] + cprev * ai;"),
    ("Thomas y' operand", "yp[i] = (y[i] - yprev * ai) / den;", "yp[i] = (y[i] - yprev * ci) / den;"),
    ("Thomas back index", "for (int i = N - 2; i >= 0; --i) u[i] = yp[i] - cp[i] * u[i + 1];",
     "for (int i = N - 2; i >= 0; --i) u[i] = yp[i] - cp[i + 1] * u[i + 1];"),
]


def _pins():
    """A fast subset of the pins; returns normally only if every one passes."""
    for N in (3, 7, 16):
        for kind in ("dd", "s1"):
            T.test_noncyclic_matches_lapack(N, kind)
    for N in (5, 6, 9, 64):
        for kind in ("dd", "s0.5"):
            T.test_cyclic_matches_lapack(N, kind)
    T.test_hyperdiffusion_discrete_amplification()
    T.test_ch_mass_conservation()
    T.test_ch_linearised_single_mode()
    T.test_ch_one_nonlinear_step_closed_form(60, 0.3)
    T.test_cn_discrete_amplification()
    T.test_cn_conserves_mean_and_matches_one_step_by_hand()
    for N in (2, 5, 33):
        T.test_thomas_matches_lapack(N, "dd")
    T.test_thomas_dirichlet_eigenmodes()
    T.test_manufactured_solution_persys(False)
    T.test_manufactured_solution_persys(True)


def _load_mutant(src_text, tmp):
    path = os.path.join(tmp, "pent_oracle_mutant.c")
    with open(path, "w") as fh:
        fh.write(src_text)
    so = os.path.join(tmp, "libmutant.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", path, "-o", so,
                    "-lm"], check=True, capture_output=True)
    return so


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, monkeypatch):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found: {old}"
    with tempfile.TemporaryDirectory() as tmp:
        so = _load_mutant(text.replace(old, new), tmp)
        real = oracle._load()
        mutant = ctypes.CDLL(so)
        for fn in dir(real):
            if fn.startswith("oracle_"):
                f_real, f_mut = getattr(real, fn), getattr(mutant, fn)
                f_mut.argtypes, f_mut.restype = f_real.argtypes, f_real.restype
        monkeypatch.setattr(oracle, "_lib", mutant)
        with np.errstate(all="ignore"):
            with pytest.raises((AssertionError, oracle.OracleError)):
                _pins()


def test_unmutated_oracle_passes_subset():
    _pins()

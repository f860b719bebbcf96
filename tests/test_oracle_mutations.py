"""The oracle's pins must catch plausible slips.

Each case plants one mistake in a copy of the C oracle on the CPU: a dropped
term, a wrong sign or index, a transposed operand, or a read before the
write.  The copy is compiled, and at least one pin must fail on it.  The real
oracle is never modified.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import reference as ref

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTATIONS = {
    "dropped_beta": ("p[j] = bt * (vt[j] - p[j]);", "p[j] = (vt[j] - p[j]);"),
    "sign_of_residual": ("p[j] = bt * (vt[j] - p[j]);", "p[j] = bt * (vt[j] + p[j]);"),
    "dropped_scale": ("const double qi = qt[i] * scale;", "const double qi = qt[i];"),
    "gate_sign": ("const double s = exp(g[tok]);", "const double s = exp(-g[tok]);"),
    "kda_gate_on_value_axis": ("for (long j = 0; j < dv; ++j) hi[j] *= a[i];",
                               "for (long j = 0; j < dv; ++j) hi[j] *= a[j % dk];"),
    "kda_first_channel_only": ("a[i] = exp(g[tok * dk + i]);", "a[i] = exp(g[tok * dk]);"),
    "predict_with_query": ("for (long j = 0; j < dv; ++j) p[j] += hi[j] * ki;",
                           "for (long j = 0; j < dv; ++j) p[j] += hi[j] * qt[i];"),
    "write_with_query": ("for (long j = 0; j < dv; ++j) hi[j] += ki * p[j];",
                         "for (long j = 0; j < dv; ++j) hi[j] += qt[i] * p[j];"),
    "decay_not_applied": ("for (long j = 0; j < dv; ++j) hi[j] *= a[i];", "(void)hi;"),
}


def _build_mutant(tmp, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = os.path.join(tmp, "mut.c")
    open(path, "w").write(src.replace(old, new))
    lib = os.path.join(tmp, "libmut.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", "-o", lib, path, "-lm"],
                   check=True)
    return lib


def _read_before_write_mutant(tmp):
    # move the read (o = scale h^T q) in front of the predict/write steps
    src = open(SRC).read()
    read_start = src.index("        /* read after the write")
    read_end = src.index("    }\n    if (hT)")
    read_block = src[read_start:read_end]
    pred_start = src.index("        /* predict with the decayed state")
    src = src[:read_start] + src[read_end:]
    src = src[:pred_start] + read_block + src[pred_start:]
    path = os.path.join(tmp, "mut.c")
    open(path, "w").write(src)
    lib = os.path.join(tmp, "libmut.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", lib, path, "-lm"], check=True)
    return lib


def _pins_pass():
    """A compact battery of the pins in test_oracle_pins.py; True if all hold."""
    rng = np.random.default_rng(0)
    B, T, H, dk, dv = 1, 9, 2, 5, 3
    q = rng.standard_normal((B, T, H, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.1, 0.9, (B, T, H))
    S0 = rng.standard_normal((B, H, dk, dv))
    ok = True
    for g in (-rng.uniform(0, 1, (B, T, H)), -rng.uniform(0, 1, (B, T, H, dk))):
        o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.7, S0)
        o2, s2 = ref.matrix_recurrence(q, k, v, g, beta, 0.7, S0)
        ok &= bool(np.allclose(o1, o2, atol=1e-12) and np.allclose(s1, s2, atol=1e-12))
        o3, _ = oracle.recurrence(k, k, v, g, np.ones_like(beta), 1.0, S0)
        ok &= bool(np.abs(o3 - v).max() < 1e-12)
    return ok


@pytest.fixture
def swap_oracle_lib():
    saved = oracle._lib
    yield
    oracle._lib = saved


def _load_into_oracle(libpath):
    lib = ctypes.CDLL(libpath)
    d = ctypes.POINTER(ctypes.c_double)
    i32 = ctypes.POINTER(ctypes.c_int)
    lib.gdn_oracle_forward.restype = ctypes.c_int
    lib.gdn_oracle_forward.argtypes = [d, d, d, d, d, ctypes.c_double, d, d, d, i32, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int]
    oracle._lib = lib


def test_unmutated_oracle_passes_battery():
    assert _pins_pass()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS) + ["read_before_write"])
def test_pins_catch_mutation(name, swap_oracle_lib):
    oracle.load()
    with tempfile.TemporaryDirectory() as tmp:
        if name == "read_before_write":
            lib = _read_before_write_mutant(tmp)
        else:
            lib = _build_mutant(tmp, *MUTATIONS[name])
        _load_into_oracle(lib)
        assert not _pins_pass(), f"mutation {name} went unnoticed"

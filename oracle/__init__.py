"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline
leg and the reference arm) may import this package.  The library's product path
never calls it, and the two share no code: the oracle is an independent
restatement of the pages, written to check the CUDA kernels.

Contents:
* ``recurrence``: the token-by-token recurrence in C (``gdn_oracle.c``), fp64,
  OpenMP over independent (sequence, head) chains.  This is the oracle the GPU
  results are compared with.  It handles the scalar gate (GDN) and the
  per-key-channel gate (KDA).  The decode step is the same recurrence, one
  token per call.
* ``recurrence_backward``: the gradients of <dO, o> + <dhT, h_final> with respect
  to q, k, v, g, beta and the initial state, by reverse-mode differentiation of
  the same token steps (C, fp64).
* ``gate_activation``, ``beta_activation``, ``activation_backward``: the gate and
  beta activations from raw logits and their chain rule (numpy, fp64).
* ``reference``: numpy twins that pin the oracle.  They are the literal d x d
  matrix recurrence, the DeltaNet and Mamba2 limits, and brute-force
  chunkwise / WY / UT evaluators with three triangular solves.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
facts the pages and the mathematics fix.  One value is parity unpinned: the
absolute output of the five configurations.  The pages print no input or
output values for them, only error magnitudes.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

__all__ = ["recurrence", "recurrence_backward", "gate_activation", "beta_activation", "activation_backward", "load",
           "max_threads"]

_lib = None


def load():
    """Build (if needed) and load the C oracle."""
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        d = ctypes.POINTER(ctypes.c_double)
        i32 = ctypes.POINTER(ctypes.c_int)
        lib.gdn_oracle_forward.restype = ctypes.c_int
        lib.gdn_oracle_forward.argtypes = [d, d, d, d, d, ctypes.c_double, d, d, d, i32, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int]
        lib.gdn_oracle_backward.restype = ctypes.c_int
        lib.gdn_oracle_backward.argtypes = [d, d, d, d, d, ctypes.c_double, d, d, d, d, d, d, d, d, d, i32,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(load().gdn_oracle_max_threads())


def _f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor (bf16/fp32) or array to a contiguous fp64 numpy array."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, g, beta, scale: float, initial_state=None, cu_seqlens=None,
               gate_per_channel: Optional[bool] = None, n_threads: int = 0):
    """Run the fp64 token recurrence.

    Shapes: q, k [B, T, H, dk]; v [B, T, H, dv]; g [B, T, H] (GDN) or
    [B, T, H, dk] (KDA); beta [B, T, H]; initial_state [N, H, dk, dv] or None;
    cu_seqlens int [n+1] or None (then B must be 1).
    Returns (o [B, T, H, dv], final_state [N, H, dk, dv]) as fp64 numpy arrays.
    """
    qd, kd, vd, gd, bd = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = qd.shape
    dv = vd.shape[-1]
    if gate_per_channel is None:
        gate_per_channel = gd.ndim == 4
    cu = None
    N = B
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    h0 = _f64(initial_state)
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = load().gdn_oracle_forward(
        _ptr(qd), _ptr(kd), _ptr(vd), _ptr(gd), _ptr(bd), float(scale), _ptr(h0), _ptr(o), _ptr(hT),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)) if cu is not None else ctypes.POINTER(ctypes.c_int)(),
        int(N if cu is not None else 0), B, T, H, dk, dv, int(bool(gate_per_channel)), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return o, hT


def recurrence_backward(q, k, v, g, beta, scale: float, d_out, initial_state=None, d_final_state=None,
                        cu_seqlens=None, gate_per_channel: Optional[bool] = None, n_threads: int = 0):
    """Gradients of L = <d_out, o> + <d_final_state, final_state> through the fp64 token recurrence.

    Shapes as ``recurrence``; d_out [B, T, H, dv]; d_final_state [N, H, dk, dv] or None (zero).
    Returns a dict of fp64 numpy arrays: dq, dk [B, T, H, dk]; dv [B, T, H, dv]; dg (the shape of g);
    dbeta [B, T, H]; dh0 [N, H, dk, dv].
    """
    qd, kd, vd, gd, bd, dod = (_f64(x) for x in (q, k, v, g, beta, d_out))
    B, T, H, dk = qd.shape
    dv = vd.shape[-1]
    if gate_per_channel is None:
        gate_per_channel = gd.ndim == 4
    cu = None
    N = B
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    h0 = _f64(initial_state)
    dhT = _f64(d_final_state)
    out = {"dq": np.zeros_like(qd), "dk": np.zeros_like(kd), "dv": np.zeros_like(vd), "dg": np.zeros_like(gd),
           "dbeta": np.zeros_like(bd), "dh0": np.zeros((N, H, dk, dv), dtype=np.float64)}
    rc = load().gdn_oracle_backward(
        _ptr(qd), _ptr(kd), _ptr(vd), _ptr(gd), _ptr(bd), float(scale), _ptr(h0), _ptr(dod), _ptr(dhT),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)) if cu is not None else ctypes.POINTER(ctypes.c_int)(),
        int(N if cu is not None else 0), B, T, H, dk, dv, int(bool(gate_per_channel)), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def _sigmoid(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def gate_activation(x, A_log, dt_bias=None):
    """log alpha = -exp(A_log[h]) softplus(x + dt_bias[h]) ("Gated Delta Network (GDN)", §3.1 eq. 5), fp64.
    x [..., H] (the head axis last); A_log, dt_bias [H]."""
    y = _f64(x) + (0.0 if dt_bias is None else _f64(dt_bias))
    return -np.exp(_f64(A_log)) * np.logaddexp(0.0, y)


def beta_activation(b, mult: int = 1):
    """beta = mult * sigmoid(b): mult 1, or 2 for beta in (0, 2) ("Gated Delta Network (GDN)", §5 notes), fp64."""
    return mult * _sigmoid(_f64(b))


def activation_backward(x, b, A_log, dt_bias, mult, dg, dbeta):
    """The chain rule through the two activations, fp64.

    With y = x + dt_bias and log alpha = -exp(A_log) softplus(y):  d log alpha / dx = -exp(A_log) sigmoid(y),
    d log alpha / dA_log = log alpha, d log alpha / d dt_bias = d log alpha / dx; with beta = mult sigmoid(b):
    d beta / db = mult sigmoid(b) (1 - sigmoid(b)).  dg, dbeta are the gradients of log alpha and beta; A_log = None
    skips the gate (dx = dg), mult = 0 skips beta (db = dbeta).  Returns dict(dx, db, dA_log [H], ddt_bias [H])."""
    dg, dbeta = _f64(dg), _f64(dbeta)
    out = {}
    if A_log is not None:
        y = _f64(x) + (0.0 if dt_bias is None else _f64(dt_bias))
        e = np.exp(_f64(A_log))
        g = -e * np.logaddexp(0.0, y)
        dx = dg * (-e * _sigmoid(y))
        axes = tuple(range(dx.ndim - 1))
        out["dx"] = dx
        out["dA_log"] = np.sum(dg * g, axis=axes)
        out["ddt_bias"] = np.sum(dx, axis=axes)
    else:
        out["dx"] = dg
    if mult:
        sb = _sigmoid(_f64(b))
        out["db"] = dbeta * mult * sb * (1.0 - sb)
    else:
        out["db"] = dbeta
    return out

"""ctypes binding of libgdn_gb300.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  torch is
used for device memory and streams.  If the library is missing, the calls
raise; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_LIB = None

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_CUDA",
                4: "GDN_ERR_TIMEOUT", 5: "GDN_ERR_NONFINITE"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}
ALGOS = {"auto": 0, "generic": 1, "tcgen05": 2, "two_pass": 3}


class GateAct(ctypes.Structure):
    """C struct gdn_gate_act: the in-kernel gate / beta activation."""
    _fields_ = [("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("beta_sigmoid", ctypes.c_int)]


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _declare(lib):
    vp, fp, i = ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    chunk = [vp, vp, vp, vp, vp, fp, vp, i, vp, vp, i, vp, i, i, i, i, i, i, i, i]
    for name in ("gdn_chunk_fwd", "kda_chunk_fwd"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i, chunk + [vp]
    for name in ("gdn_chunk_fwd_algo", "kda_chunk_fwd_algo"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i, chunk + [i, vp]
    for name in ("gdn_chunk_fwd_ws", "kda_chunk_fwd_ws"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i, chunk + [i, vp, ctypes.c_size_t, vp]
    lib.gdn_chunk_fwd_ex.restype = i
    lib.gdn_chunk_fwd_ex.argtypes = [i] + chunk[:14] + [i] + chunk[14:] + [ctypes.POINTER(GateAct), i, vp,
                                                                           ctypes.c_size_t, vp]
    lib.gdn_recurrent_step_ex.restype = i
    lib.gdn_recurrent_step_ex.argtypes = [i, vp, vp, vp, vp, vp, fp, vp, vp, i, i, i, i, i, i, i,
                                          ctypes.POINTER(GateAct), vp]
    lib.gdn_chunk_fwd_act.restype = i
    lib.gdn_chunk_fwd_act.argtypes = chunk + [ctypes.POINTER(GateAct), i, vp, ctypes.c_size_t, vp]
    lib.gdn_recurrent_step_act.restype = i
    lib.gdn_recurrent_step_act.argtypes = [vp, vp, vp, vp, vp, fp, vp, vp, i, i, i, i, i, i,
                                           ctypes.POINTER(GateAct), vp]
    lib.gdn_chunk_fwd_noalloc.restype = i
    lib.gdn_chunk_fwd_noalloc.argtypes = [i] + chunk + [vp]
    lib.gdn_chunk_workspace_size.restype = i
    lib.gdn_chunk_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    for name in ("gdn_recurrent_step", "kda_recurrent_step"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i, [vp, vp, vp, vp, vp, fp, vp, vp, i, i, i, i, i, i, vp]
    lib.gdn_chunk_plan.restype = i
    lib.gdn_chunk_plan.argtypes = [i, i, i, i, i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_chunk_bwd.restype = i
    lib.gdn_chunk_bwd.argtypes = [i, vp, vp, vp, vp, vp, fp, vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp,
                                  i, i, i, i, i, i, i, i, vp, ctypes.c_size_t, vp]
    lib.gdn_chunk_bwd_act.restype = i
    lib.gdn_chunk_bwd_act.argtypes = [i, vp, vp, vp, vp, vp, fp, vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, vp,
                                      i, i, i, i, i, i, i, i, ctypes.POINTER(GateAct), vp, ctypes.c_size_t, vp]
    lib.gdn_chunk_bwd_ex.restype = i
    lib.gdn_chunk_bwd_ex.argtypes = [i, vp, vp, vp, vp, vp, fp, vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, vp,
                                     i, i, i, i, i, i, i, i, i, ctypes.POINTER(GateAct), vp, ctypes.c_size_t, vp]
    lib.gdn_chunk_bwd_workspace_size_ex.restype = i
    lib.gdn_chunk_bwd_workspace_size_ex.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.gdn_chunk_bwd_workspace_size.restype = i
    lib.gdn_chunk_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.gdn_test_inject.restype = i
    lib.gdn_test_inject.argtypes = [i]
    lib.gdn_last_error.argtypes = []
    lib.gdn_device_status.restype = i
    lib.gdn_device_status.argtypes = [i]
    lib.gdn_version.restype = ctypes.c_char_p
    lib.gdn_version.argtypes = []
    return lib


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libgdn_gb300.so (built by gated_delta_rule_gdn_gb300.build.build()); raise if missing."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libgdn_gb300.so is not built ({path}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        _LIB = _declare(ctypes.CDLL(path))
    return _LIB


def last_error() -> str:
    return load().gdn_last_error().decode()


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, last_error())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def workspace_size(per_channel: bool, B: int, T: int, H: int, dk: int, dv: int, chunk_size: int, dtype,
                   n_seqs: int = 0, algo: str = "auto", o_dtype=torch.float32) -> int:
    """Device workspace bytes a chunk-forward call with these sizes needs (0 if its kernel needs none)."""
    out = ctypes.c_size_t(0)
    _check(load().gdn_chunk_workspace_size(int(per_channel), B, T, H, dk, dv, chunk_size, DTYPES[dtype],
                                           DTYPES[o_dtype], int(n_seqs), ALGOS[algo], ctypes.byref(out)))
    return int(out.value)


def _gate_act(dev, H, A_log, dt_bias, beta_sigmoid, allow_neg_eigval=False):
    """The activation descriptor (or None) after checking its tensors.  With ``allow_neg_eigval`` the sigmoid of
    beta is doubled (beta in (0, 2))."""
    if allow_neg_eigval and not beta_sigmoid:
        raise ValueError("allow_neg_eigval scales the in-kernel sigmoid of beta: it needs beta_sigmoid")
    if A_log is None and dt_bias is None and not beta_sigmoid:
        return None
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias)):
        if t is not None:
            _need(t, name, torch.float32, dev)
            if t.shape != (H,):
                raise ValueError(f"{name} must have shape ({H},)")
    return GateAct(None if A_log is None else A_log.data_ptr(), None if dt_bias is None else dt_bias.data_ptr(),
                   (2 if allow_neg_eigval else 1) if beta_sigmoid else 0)


def _chunk(per_channel: bool, q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
           cu_seqlens=None, chunk_size=64, algo="auto", o=None, final_state=None, stream=None,
           o_dtype=torch.float32, workspace=None, A_log=None, dt_bias=None, beta_sigmoid=False,
           allow_neg_eigval=False):
    lib = load()
    if q.dtype not in DTYPES:
        raise ValueError(f"q must be float32 or bfloat16 (got {q.dtype})")
    dev = q.device
    for name, t, dt in (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype), ("g", g, torch.float32),
                        ("beta", beta, torch.float32)):
        _need(t, name, dt, dev)
    B, T, Hk, dk = q.shape
    H = v.shape[2]            # value heads (a multiple of the key heads of q and k)
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:2] != (B, T) or H % Hk != 0:
        raise ValueError("q, k, v shapes do not match")
    if g.shape != ((B, T, H, dk) if per_channel else (B, T, H)) or beta.shape != (B, T, H):
        raise ValueError("g / beta shapes do not match")
    n_seqs = 0
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        n_seqs = cu_seqlens.numel() - 1
    N = n_seqs if cu_seqlens is not None else B
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev)
        if initial_state.shape != (N, H, dk, dv):
            raise ValueError(f"initial_state must be {(N, H, dk, dv)}")
    if o_dtype not in DTYPES:
        raise ValueError(f"o_dtype must be float32 or bfloat16 (got {o_dtype})")
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=o_dtype, device=dev)
    _need(o, "o", o_dtype, dev)
    if output_final_state and final_state is None:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, dev)
    if scale is None:
        scale = dk ** -0.5
    if workspace is None:
        need = workspace_size(per_channel, B, T, H, dk, dv, int(chunk_size), q.dtype, n_seqs, algo, o_dtype)
        if need > 0:
            # torch's caching allocator keeps the block for the next call
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev)
    act = _gate_act(dev, H, A_log, dt_bias, beta_sigmoid, allow_neg_eigval)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(initial_state),
            int(final_state is not None), _ptr(final_state), _ptr(cu_seqlens), n_seqs, _ptr(o),
            B, T, H, dk, dv, int(chunk_size), DTYPES[q.dtype], DTYPES[o_dtype])
    tail = (ALGOS[algo], _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream_handle(stream, dev))
    if act is not None or Hk != H:
        ext = args[:14] + (Hk,) + args[14:]
        st = lib.gdn_chunk_fwd_ex(int(per_channel), *ext, None if act is None else ctypes.byref(act), *tail)
    else:
        fn = lib.kda_chunk_fwd_ws if per_channel else lib.gdn_chunk_fwd_ws
        st = fn(*args, *tail)
    _check(st)
    return o, final_state


def gdn_chunk_fwd(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False, cu_seqlens=None,
                  chunk_size=64, algo="auto", o=None, final_state=None, stream=None, o_dtype=torch.float32,
                  workspace=None, A_log=None, dt_bias=None, beta_sigmoid=False, allow_neg_eigval=False):
    """Chunkwise gated delta rule forward (C ABI gdn_chunk_fwd_ws, or gdn_chunk_fwd_act with an activation).
    Returns (o, final_state or None).

    o is fp32 unless o_dtype=torch.bfloat16 (then it is the round-to-nearest-even of the fp32 result).
    ``workspace`` (uint8 device tensor, see workspace_size) is allocated here when the kernel needs one.
    ``A_log``/``dt_bias`` ([H] fp32): g holds raw logits and the kernel applies -exp(A_log) softplus(g + dt_bias);
    ``beta_sigmoid``: beta holds logits (sigmoid in the kernel; 2 sigmoid, beta in (0, 2), with
    ``allow_neg_eigval``).  q and k may have fewer heads than v (grouped value heads).
    """
    return _chunk(False, q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens, chunk_size, algo,
                  o, final_state, stream, o_dtype, workspace, A_log, dt_bias, beta_sigmoid, allow_neg_eigval)


def kda_chunk_fwd(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False, cu_seqlens=None,
                  chunk_size=64, algo="auto", o=None, final_state=None, stream=None, o_dtype=torch.float32,
                  workspace=None, beta_sigmoid=False, allow_neg_eigval=False):
    """Chunkwise KDA forward, g per key channel (C ABI kda_chunk_fwd_ws).  Returns (o, final_state or None).
    ``beta_sigmoid``/``allow_neg_eigval`` as for gdn_chunk_fwd; the gate itself is taken as given."""
    return _chunk(True, q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens, chunk_size, algo,
                  o, final_state, stream, o_dtype, workspace, None, None, beta_sigmoid, allow_neg_eigval)


def chunk_fwd_noalloc(per_channel: bool, q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                      cu_seqlens=None, o=None, final_state=None, stream=None, o_dtype=torch.float32):
    """The two-pass chunk forward with the library's static scratch (C ABI gdn_chunk_fwd_noalloc): no allocation
    inside the call.  Returns (o, final_state or None); raises GdnError for requests above the scratch limit."""
    lib = load()
    dev = q.device
    for name, t, dt in (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype), ("g", g, torch.float32),
                        ("beta", beta, torch.float32)):
        _need(t, name, dt, dev)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    n_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    N = n_seqs if cu_seqlens is not None else B
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=o_dtype, device=dev)
    if output_final_state and final_state is None:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if scale is None:
        scale = dk ** -0.5
    st = lib.gdn_chunk_fwd_noalloc(int(per_channel), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                   _ptr(initial_state), int(final_state is not None), _ptr(final_state),
                                   _ptr(cu_seqlens), n_seqs, _ptr(o), B, T, H, dk, dv, 64, DTYPES[q.dtype],
                                   DTYPES[o_dtype], _stream_handle(stream, dev))
    _check(st)
    return o, final_state


def bwd_workspace_size(per_channel: bool, B: int, T: int, H: int, dk: int, dv: int, chunk_size: int = 0,
                       n_seqs: int = 0, Hk: int = 0) -> int:
    """Device workspace bytes of a chunk-backward call (C ABI gdn_chunk_bwd_workspace_size_ex; Hk key heads, 0: H)."""
    out = ctypes.c_size_t(0)
    _check(load().gdn_chunk_bwd_workspace_size_ex(int(per_channel), B, T, int(Hk), H, dk, dv, int(chunk_size),
                                                  int(n_seqs), ctypes.byref(out)))
    return int(out.value)


def chunk_bwd(per_channel: bool, q, k, v, g, beta, d_o, scale=None, initial_state=None, d_final_state=None,
              cu_seqlens=None, chunk_size=0, stream=None, workspace=None, want_d_initial_state=True, A_log=None,
              dt_bias=None, beta_sigmoid=False, allow_neg_eigval=False):
    """Gradients of <d_o, o> + <d_final_state, final_state> through the chunk forward (C ABI gdn_chunk_bwd, or
    gdn_chunk_bwd_act with an activation).

    Inputs as the forward (per_channel: KDA gate [B, T, H, dk]); d_o [B, T, H, dv] fp32 or bf16; d_final_state
    [N, H, dk, dv] fp32 or None.  Returns (dq, dk, dv, dg, dbeta, d_initial_state or None), all fp32.  With
    A_log / dt_bias / beta_sigmoid as for gdn_chunk_fwd, g and beta are raw logits, dg and dbeta are their
    gradients, and the result gains (dA_log, ddt_bias or None) at the end."""
    lib = load()
    if q.dtype not in DTYPES:
        raise ValueError(f"q must be float32 or bfloat16 (got {q.dtype})")
    dev = q.device
    for name, t, dt in (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype), ("g", g, torch.float32),
                        ("beta", beta, torch.float32), ("d_o", d_o, None)):
        _need(t, name, dt, dev)
    if d_o.dtype not in DTYPES:
        raise ValueError(f"d_o must be float32 or bfloat16 (got {d_o.dtype})")
    B, T, Hk, dk = q.shape
    H = v.shape[2]            # value heads (a multiple of the key heads of q and k)
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:2] != (B, T) or H % Hk != 0 or d_o.shape != v.shape:
        raise ValueError("q, k, v, d_o shapes do not match")
    if g.shape != ((B, T, H, dk) if per_channel else (B, T, H)) or beta.shape != (B, T, H):
        raise ValueError("g / beta shapes do not match")
    n_seqs = 0
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        n_seqs = cu_seqlens.numel() - 1
    N = n_seqs if cu_seqlens is not None else B
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _need(t, name, torch.float32, dev)
            if t.shape != (N, H, dk, dv):
                raise ValueError(f"{name} must be {(N, H, dk, dv)}")
    if scale is None:
        scale = dk ** -0.5
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dkk, dvv = torch.empty(q.shape, **f32), torch.empty(k.shape, **f32), torch.empty(v.shape, **f32)
    dg, dbeta = torch.empty(g.shape, **f32), torch.empty(beta.shape, **f32)
    dh0 = torch.empty((N, H, dk, dv), **f32) if want_d_initial_state else None
    if workspace is None:
        need = bwd_workspace_size(per_channel, B, T, H, dk, dv, chunk_size, n_seqs, Hk)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev)
    act = _gate_act(dev, H, A_log, dt_bias, beta_sigmoid, allow_neg_eigval)
    dA = torch.empty(H, **f32) if A_log is not None else None
    ddt = torch.empty(H, **f32) if dt_bias is not None else None
    _check(lib.gdn_chunk_bwd_ex(int(per_channel), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                _ptr(initial_state), _ptr(d_o), _ptr(d_final_state), _ptr(cu_seqlens), n_seqs,
                                _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(dA),
                                _ptr(ddt), B, T, Hk, H, dk, dv, int(chunk_size), DTYPES[q.dtype], DTYPES[d_o.dtype],
                                None if act is None else ctypes.byref(act), _ptr(workspace),
                                0 if workspace is None else workspace.numel(), _stream_handle(stream, dev)))
    if act is None:
        return dq, dkk, dvv, dg, dbeta, dh0
    return dq, dkk, dvv, dg, dbeta, dh0, dA, ddt


def gdn_chunk_bwd(q, k, v, g, beta, d_o, **kw):
    """Backward of gdn_chunk_fwd (scalar gate): see chunk_bwd."""
    return chunk_bwd(False, q, k, v, g, beta, d_o, **kw)


def kda_chunk_bwd(q, k, v, g, beta, d_o, **kw):
    """Backward of kda_chunk_fwd (per-channel gate): see chunk_bwd."""
    return chunk_bwd(True, q, k, v, g, beta, d_o, **kw)


def _step(per_channel: bool, q, k, v, g, beta, state, scale=None, o=None, stream=None, o_dtype=torch.float32,
          A_log=None, dt_bias=None, beta_sigmoid=False, allow_neg_eigval=False):
    lib = load()
    if q.dtype not in DTYPES:
        raise ValueError(f"q must be float32 or bfloat16 (got {q.dtype})")
    dev = q.device
    for name, t, dt in (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype), ("g", g, torch.float32),
                        ("beta", beta, torch.float32), ("state", state, torch.float32)):
        _need(t, name, dt, dev)
    N, Hk, dk = q.shape
    H = v.shape[1]            # value heads (a multiple of the key heads of q and k)
    dv = v.shape[-1]
    g_shape = (N, H, dk) if per_channel else (N, H)
    if (state.shape != (N, H, dk, dv) or k.shape != q.shape or g.shape != g_shape or beta.shape != (N, H)
            or H % Hk != 0):
        raise ValueError("decode shapes do not match")
    if o_dtype not in DTYPES:
        raise ValueError(f"o_dtype must be float32 or bfloat16 (got {o_dtype})")
    if o is None:
        o = torch.empty((N, H, dv), dtype=o_dtype, device=dev)
    _need(o, "o", o_dtype, dev)
    if scale is None:
        scale = dk ** -0.5
    act = _gate_act(dev, H, A_log, dt_bias, beta_sigmoid, allow_neg_eigval)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(state), _ptr(o), N, H, dk, dv,
            DTYPES[q.dtype], DTYPES[o_dtype])
    if act is not None or Hk != H:
        ext = args[:8] + (N, Hk) + args[9:]
        st = lib.gdn_recurrent_step_ex(int(per_channel), *ext, None if act is None else ctypes.byref(act),
                                       _stream_handle(stream, dev))
    else:
        fn = lib.kda_recurrent_step if per_channel else lib.gdn_recurrent_step
        st = fn(*args, _stream_handle(stream, dev))
    _check(st)
    return o


def gdn_recurrent_step(q, k, v, g, beta, state, scale=None, o=None, stream=None, o_dtype=torch.float32,
                       A_log=None, dt_bias=None, beta_sigmoid=False, allow_neg_eigval=False):
    """One decode token for N sequences (C ABI gdn_recurrent_step, or gdn_recurrent_step_act with an activation);
    updates ``state`` in place, returns o."""
    return _step(False, q, k, v, g, beta, state, scale, o, stream, o_dtype, A_log, dt_bias, beta_sigmoid,
                 allow_neg_eigval)


def kda_recurrent_step(q, k, v, g, beta, state, scale=None, o=None, stream=None, o_dtype=torch.float32,
                       beta_sigmoid=False, allow_neg_eigval=False):
    """One KDA decode token, g per key channel [N, H, d_k] (C ABI kda_recurrent_step); updates ``state`` in place."""
    return _step(True, q, k, v, g, beta, state, scale, o, stream, o_dtype, None, None, beta_sigmoid,
                 allow_neg_eigval)


def chunk_plan(per_channel: bool, B: int, T: int, H: int, dk: int, dv: int, chunk_size: int, dtype,
               varlen: bool = False, algo: str = "auto", o_dtype=torch.float32) -> str:
    """Name of the kernel ("generic" or "two_pass") a chunk-forward call with these sizes runs."""
    out = ctypes.c_int(-1)
    _check(load().gdn_chunk_plan(int(per_channel), B, T, H, dk, dv, chunk_size, DTYPES[dtype], DTYPES[o_dtype],
                                 int(varlen), ALGOS[algo], ctypes.byref(out)))
    return {v: k for k, v in ALGOS.items()}[out.value]


def device_status(clear: bool = True) -> int:
    """GDN_OK; GDN_ERR_TIMEOUT if a kernel gave up a bounded wait; GDN_ERR_NONFINITE if a chunk forward wrote a
    non-finite value to o or the final state (synchronises the device)."""
    return int(load().gdn_device_status(int(clear)))

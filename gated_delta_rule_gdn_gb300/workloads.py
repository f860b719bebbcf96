"""Seeded synthetic inputs for the gated delta rule workloads.

This module only draws inputs.  It holds none of the method's arithmetic, so
both the CUDA path and the fp64 oracle can take their inputs from it.

Random numbers come from numpy's PCG64 ``Generator``.  Its streams are the
same on x86_64 and aarch64 hosts, so a seed fixes the inputs on every machine.
The draw order of every recipe is fixed and written out below.  Tensors are
returned as CPU ``torch`` tensors in the dtype the library takes:
* q, k, v in bf16 or fp32;
* g (log retention), beta and the states in fp32;
* cu_seqlens in int32.

The value recipes come from the gated delta rule pages.  They are synthetic
stand-ins for model activations: no dataset or trained weights are involved.
* q, k ~ N(0, 1), then L2-normalised per token over d_k in fp32, then rounded
  to the storage dtype.
* v ~ N(0, 1).
* beta = sigmoid(N(0, 1)).
* GDN gate: log alpha = -A_h * softplus(N(0, 1) + dt_bias_h), with
  A_h ~ U(0, 16) and dt_bias_h ~ N(0, 0.1) drawn once per head.  This is the
  Mamba2-style parameterisation on the page "Gated Delta Network (GDN)",
  §3.1, eq. 5.
* KDA gate: log gamma = -exp(N(0, 0.5)) * softplus(N(0, 1)), per key channel.
* Initial states ~ N(0, sigma), where sigma is a standard deviation.
* Upstream gradients of a backward problem: dO ~ N(0, 1) in the storage dtype,
  and the final-state gradient ~ N(0, sigma) in fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

__all__ = [
    "ChunkWorkload", "DecodeWorkload", "CONFIGS", "chunk_inputs", "chunk_output_grads", "decode_constants",
    "decode_step_inputs", "varlen_lengths", "config", "HEAD256",
]


@dataclasses.dataclass(frozen=True)
class ChunkWorkload:
    """A chunk-forward problem: shapes, dtype and value recipe."""
    name: str
    kind: str                 # "gdn" (scalar gate per head) or "kda" (per-key-channel gate)
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk_size: int
    dtype: str                # "bf16" or "f32" for q, k, v, o
    h0_std: float = 0.0       # 0 -> no initial state (zeros)
    output_final_state: bool = True
    n_seqs: int = 0           # > 0 -> packed variable-length input (B must be 1)
    len_lo: int = 0           # range the sequence lengths are drawn from
    len_hi: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)

    @property
    def tokens(self) -> int:
        return self.B * self.T


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """A fused recurrent decode problem: N independent sequences, one token per step."""
    name: str
    N: int
    H: int
    dk: int
    dv: int
    steps: int
    dtype: str = "bf16"
    h0_std: float = 0.02
    kind: str = "gdn"         # "gdn" (scalar gate per head) or "kda" (per-key-channel gate)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)


CONFIGS = {
    0: ChunkWorkload("gdn_tiny_b1_t64_h1_d16_c16_f32", "gdn", 1, 64, 1, 16, 16, 16, "f32", h0_std=0.0),
    1: ChunkWorkload("gdn_prefill_b4_t4096_h16_d128_c64_bf16", "gdn", 4, 4096, 16, 128, 128, 64, "bf16",
                     h0_std=0.02),
    2: ChunkWorkload("gdn_varlen_8seq_65536tok_h32_d128_c64_bf16", "gdn", 1, 65536, 32, 128, 128, 64, "bf16",
                     h0_std=0.02, n_seqs=8, len_lo=256, len_hi=16384),
    3: ChunkWorkload("kda_b2_t8192_h32_d128_c64_bf16", "kda", 2, 8192, 32, 128, 128, 64, "bf16", h0_std=0.0),
    4: DecodeWorkload("decode_n256_h32_d128_1024steps", 256, 32, 128, 128, 1024),
}


# Head size 256, the largest the gated delta rule's head-size range allows ("Gated Delta Network (GDN)", §4.3), at
# the model width of config 1 (H x d = 2048).
HEAD256 = ChunkWorkload("gdn_prefill_b4_t4096_h8_d256_c64_bf16", "gdn", 4, 4096, 8, 256, 256, 64, "bf16",
                        h0_std=0.02)


def config(i: int):
    return CONFIGS[i]


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _softplus(x: np.ndarray) -> np.ndarray:
    # input synthesis only (the gate recipe); log1p(exp(x)) in a form that does not overflow
    return np.logaddexp(0.0, x)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    """L2-normalise the last axis in fp32 (the recipe's key/query normalisation)."""
    x = x.astype(np.float32, copy=False)
    n = np.sqrt(np.einsum("...i,...i->...", x, x))[..., None]
    return x / np.maximum(n, np.float32(1e-12))


def varlen_lengths(n_seqs: int, total: int, lo: int, hi: int, rng: np.random.Generator) -> np.ndarray:
    """Draw n_seqs lengths uniformly from [lo, hi], then rescale them so they sum to total.

    The scaled lengths are rounded and the rounding residual goes to the last
    length.  Each length is kept >= 1; where that clamp moves a length, the
    difference is taken back from the longest one.
    """
    raw = rng.integers(lo, hi + 1, size=n_seqs).astype(np.float64)
    lens = np.rint(raw * (total / raw.sum())).astype(np.int64)
    lens[-1] += total - lens.sum()
    lens = np.maximum(lens, 1)
    lens[np.argmax(lens)] -= lens.sum() - total
    assert lens.sum() == total and (lens >= 1).all()
    return lens


def chunk_inputs(w: ChunkWorkload, seed: int = 0, *, T: Optional[int] = None, H: Optional[int] = None,
                 B: Optional[int] = None) -> dict:
    """Draw one chunk-forward problem.

    Draw order, all from one ``np.random.default_rng(seed)``:
    1. sequence lengths (packed workloads only);
    2. q, k, v;
    3. the beta logits;
    4. the gate: for GDN, A and dt_bias per head and then the gate logits; for
       KDA, the two normal fields;
    5. the initial state, when h0_std > 0.

    ``T``, ``H`` and ``B`` override the workload's sizes (small parity cases
    that keep the same recipe).
    """
    B = w.B if B is None else B
    T = w.T if T is None else T
    H = w.H if H is None else H
    rng = np.random.default_rng(seed)
    cu = None
    N = B
    if w.n_seqs > 0:
        assert B == 1
        lens = varlen_lengths(w.n_seqs, T, w.len_lo, w.len_hi, rng)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        N = w.n_seqs
    q = _unit_rows(rng.standard_normal((B, T, H, w.dk), dtype=np.float32))
    k = _unit_rows(rng.standard_normal((B, T, H, w.dk), dtype=np.float32))
    v = rng.standard_normal((B, T, H, w.dv), dtype=np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H), dtype=np.float32).astype(np.float64))))
    if w.kind == "gdn":
        A = rng.uniform(0.0, 16.0, size=H)
        dt_bias = rng.normal(0.0, 0.1, size=H)
        logits = rng.standard_normal((B, T, H), dtype=np.float32).astype(np.float64)
        g = -A * _softplus(logits + dt_bias)
    elif w.kind == "kda":
        a = rng.standard_normal((B, T, H, w.dk), dtype=np.float32).astype(np.float64) * 0.5
        s = rng.standard_normal((B, T, H, w.dk), dtype=np.float32).astype(np.float64)
        g = -np.exp(a) * _softplus(s)
    else:
        raise ValueError(w.kind)
    h0 = None
    if w.h0_std > 0:
        h0 = (rng.standard_normal((N, H, w.dk, w.dv), dtype=np.float32) * np.float32(w.h0_std))
    dt = _torch_dtype(w.dtype)
    out = {
        "q": torch.from_numpy(q).to(dt),
        "k": torch.from_numpy(k).to(dt),
        "v": torch.from_numpy(v).to(dt),
        "g": torch.from_numpy(g.astype(np.float32)),
        "beta": torch.from_numpy(beta.astype(np.float32)),
        "initial_state": None if h0 is None else torch.from_numpy(h0),
        "cu_seqlens": None if cu is None else torch.from_numpy(cu),
        "scale": w.scale,
        "chunk_size": w.chunk_size,
        "gate_per_channel": w.kind == "kda",
        "N": N,
    }
    return out


def chunk_output_grads(x: dict, seed: int = 1, dhT_std: float = 1.0) -> dict:
    """Draw the upstream gradients for the chunk problem ``x`` (from chunk_inputs).

    From ``np.random.default_rng(seed)``, in this order: d_o ~ N(0, 1) with v's shape and dtype, then
    d_final_state ~ N(0, dhT_std) [N, H, dk, dv] fp32 (None when dhT_std is 0).
    """
    rng = np.random.default_rng(seed)
    B, T, H, dv = x["v"].shape
    dk = x["q"].shape[-1]
    d_o = rng.standard_normal((B, T, H, dv), dtype=np.float32)
    dhT = None
    if dhT_std > 0:
        dhT = rng.standard_normal((x["N"], H, dk, dv), dtype=np.float32) * np.float32(dhT_std)
    return {"d_o": torch.from_numpy(d_o).to(x["v"].dtype),
            "d_final_state": None if dhT is None else torch.from_numpy(dhT)}


def decode_constants(w: DecodeWorkload, seed: int = 0) -> dict:
    """Per-head gate constants (A, dt_bias) and the initial state, from ``default_rng(seed)``."""
    rng = np.random.default_rng(seed)
    A = rng.uniform(0.0, 16.0, size=w.H)
    dt_bias = rng.normal(0.0, 0.1, size=w.H)
    h0 = rng.standard_normal((w.N, w.H, w.dk, w.dv), dtype=np.float32) * np.float32(w.h0_std)
    return {"A": A, "dt_bias": dt_bias, "state": torch.from_numpy(h0)}


def decode_step_inputs(w: DecodeWorkload, consts: dict, step: int, seed: int = 0, n: Optional[int] = None) -> dict:
    """Inputs of decode step ``step``, drawn from ``default_rng([seed, 1000 + step])``.

    Draw order: q, k, v, beta logits, gate logits.  Shapes are [N, H, d] for
    q, k and v, [N, H] for beta, and [N, H] for g (the GDN gate) or
    [N, H, d_k] (the KDA gate, drawn as in the KDA chunk recipe:
    -exp(N(0, 0.5)) softplus(N(0, 1))).  ``n`` overrides N and keeps the
    leading rows of each draw.
    """
    N = w.N if n is None else n
    rng = np.random.default_rng([seed, 1000 + step])
    q = _unit_rows(rng.standard_normal((w.N, w.H, w.dk), dtype=np.float32))[:N]
    k = _unit_rows(rng.standard_normal((w.N, w.H, w.dk), dtype=np.float32))[:N]
    v = rng.standard_normal((w.N, w.H, w.dv), dtype=np.float32)[:N]
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((w.N, w.H), dtype=np.float32).astype(np.float64)))[:N]
    if w.kind == "kda":
        a = rng.standard_normal((w.N, w.H, w.dk), dtype=np.float32).astype(np.float64)[:N] * 0.5
        sp = rng.standard_normal((w.N, w.H, w.dk), dtype=np.float32).astype(np.float64)[:N]
        g = -np.exp(a) * _softplus(sp)
    else:
        logits = rng.standard_normal((w.N, w.H), dtype=np.float32).astype(np.float64)[:N]
        g = -consts["A"] * _softplus(logits + consts["dt_bias"])
    dt = _torch_dtype(w.dtype)
    return {
        "q": torch.from_numpy(np.ascontiguousarray(q)).to(dt),
        "k": torch.from_numpy(np.ascontiguousarray(k)).to(dt),
        "v": torch.from_numpy(np.ascontiguousarray(v)).to(dt),
        "g": torch.from_numpy(np.ascontiguousarray(g.astype(np.float32))),
        "beta": torch.from_numpy(np.ascontiguousarray(beta.astype(np.float32))),
    }

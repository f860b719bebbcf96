"""Shared helpers for the GPU-vs-oracle parity tests.

The tolerances are those the target sets for this method:
* fp32 inputs: relative L2 error <= 1e-4 for the output and the final state.
* bf16 q/k/v with fp32 gates and state: relative L2 error <= 5e-3, and
  max |error| / rms(oracle) <= 2e-2, for both tensors.
Here rel-L2 = ||x - y||_2 / ||y||_2 over the whole compared tensor.
"""
import numpy as np
import torch

import oracle

F32_REL_L2 = 1e-4
BF16_REL_L2 = 5e-3
BF16_MAX_OVER_RMS = 2e-2


def rel_l2(x: np.ndarray, y: np.ndarray) -> float:
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def max_over_rms(x: np.ndarray, y: np.ndarray) -> float:
    return float(np.abs(x - y).max() / max(np.sqrt(np.mean(y ** 2)), 1e-300))


def assert_close(x, y, dtype, what=""):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (what, x.shape, y.shape)
    assert np.isfinite(x).all(), f"{what}: non-finite values"
    e = rel_l2(x, y)
    if dtype == torch.float32:
        assert e <= F32_REL_L2, f"{what}: rel-L2 {e:.3e} > {F32_REL_L2}"
    else:
        m = max_over_rms(x, y)
        assert e <= BF16_REL_L2, f"{what}: rel-L2 {e:.3e} > {BF16_REL_L2}"
        assert m <= BF16_MAX_OVER_RMS, f"{what}: max/rms {m:.3e} > {BF16_MAX_OVER_RMS}"
    return e


def to_dev(x: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def oracle_on_heads(x: dict, heads=None):
    """Run the fp64 oracle on a subset of heads (all sequences); returns (o, final_state) for those heads."""
    q, k, v, g, beta = x["q"], x["k"], x["v"], x["g"], x["beta"]
    h0 = x["initial_state"]
    if heads is not None:
        hs = torch.as_tensor(heads)
        q, k, v, g, beta = (t.index_select(2, hs) for t in (q, k, v, g, beta))
        if h0 is not None:
            h0 = h0.index_select(1, hs)
    return oracle.recurrence(q, k, v, g, beta, x["scale"], h0, x["cu_seqlens"],
                             gate_per_channel=x["gate_per_channel"])

"""The seeded input generators: shapes, dtypes, determinism and the value recipe."""
import numpy as np
import torch

from gated_delta_rule_gdn_gb300 import workloads as W


def test_tiny_config_shapes_and_recipe():
    w = W.config(0)
    x = W.chunk_inputs(w, seed=0)
    assert x["q"].shape == (1, 64, 1, 16) and x["q"].dtype == torch.float32
    assert x["v"].shape == (1, 64, 1, 16)
    assert x["g"].shape == (1, 64, 1) and x["beta"].shape == (1, 64, 1)
    assert x["initial_state"] is None and x["cu_seqlens"] is None
    assert abs(x["scale"] - 0.25) < 1e-15
    nq = x["q"].double().norm(dim=-1)
    assert torch.allclose(nq, torch.ones_like(nq), atol=1e-6)
    assert (x["g"] <= 0).all() and ((x["beta"] > 0) & (x["beta"] < 1)).all()


def test_generation_is_deterministic():
    w = W.config(1)
    a = W.chunk_inputs(w, seed=3, T=128, H=2, B=1)
    b = W.chunk_inputs(w, seed=3, T=128, H=2, B=1)
    for key in ("q", "k", "v", "g", "beta", "initial_state"):
        assert torch.equal(a[key], b[key])
    c = W.chunk_inputs(w, seed=4, T=128, H=2, B=1)
    assert not torch.equal(a["v"], c["v"])


def test_bf16_keys_are_unit_to_bf16_precision():
    x = W.chunk_inputs(W.config(1), seed=0, T=256, H=2, B=1)
    assert x["k"].dtype == torch.bfloat16
    n = x["k"].double().norm(dim=-1)
    assert (n - 1).abs().max() < 1e-2
    assert x["initial_state"].dtype == torch.float32
    assert abs(float(x["initial_state"].std()) - 0.02) < 2e-3


def test_varlen_lengths_reading():
    rng = np.random.default_rng(0)
    lens = W.varlen_lengths(8, 65536, 256, 16384, rng)
    assert lens.sum() == 65536 and len(lens) == 8 and (lens >= 1).all()
    x = W.chunk_inputs(W.config(2), seed=0, T=4096, H=2)
    cu = x["cu_seqlens"]
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and int(cu[-1]) == 4096
    assert (cu[1:] >= cu[:-1]).all() and x["N"] == 8


def test_kda_gate_is_per_channel_and_nonpositive():
    x = W.chunk_inputs(W.config(3), seed=0, T=64, H=2, B=1)
    assert x["g"].shape == (1, 64, 2, 128) and (x["g"] <= 0).all()
    assert x["gate_per_channel"]


def test_decode_step_inputs():
    w = W.config(4)
    c = W.decode_constants(W.DecodeWorkload("t", 4, 2, 16, 8, 3), seed=0)
    assert c["state"].shape == (4, 2, 16, 8)
    s0 = W.decode_step_inputs(W.DecodeWorkload("t", 4, 2, 16, 8, 3), c, 0)
    s1 = W.decode_step_inputs(W.DecodeWorkload("t", 4, 2, 16, 8, 3), c, 1)
    assert s0["q"].shape == (4, 2, 16) and s0["v"].shape == (4, 2, 8) and s0["g"].shape == (4, 2)
    assert not torch.equal(s0["k"], s1["k"])
    assert w.N == 256 and w.steps == 1024

"""GPU parity of the decode step (gdn_recurrent_step) against the fp64 oracle.

The decode step is the token recurrence, one token per call.  So a run of S
steps must match the oracle on those S tokens:
* every step's output;
* the state after the last step.
The full-size case has 256 sequences, 32 heads and d = 128, and runs all 1024
steps.  There, the oracle follows a sample of (sequence, head) chains.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import gated_delta_rule_gdn_gb300 as gdn
import oracle
from gated_delta_rule_gdn_gb300 import workloads as W
from parity_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_gdn_gb300 import build
    build.build()
    gdn.load()


def _decode_and_compare(w: W.DecodeWorkload, steps: int, sample=None):
    consts = W.decode_constants(w, seed=0)
    state = consts["state"].cuda()
    NH = w.N * w.H
    idx = np.arange(NH) if sample is None else np.asarray(sample)
    tidx = torch.as_tensor(idx)
    h0s = consts["state"].reshape(NH, w.dk, w.dv)[tidx][:, None].clone()
    kept = {key: [] for key in ("q", "k", "v", "g", "beta")}
    outs = []
    # inputs are drawn on host threads a few steps ahead; only the sampled chains are kept for the oracle
    with cf.ThreadPoolExecutor(8) as ex:
        pending = {s: ex.submit(W.decode_step_inputs, w, consts, s) for s in range(min(steps, 16))}
        for s in range(steps):
            x = pending.pop(s).result()
            if s + 16 < steps:
                pending[s + 16] = ex.submit(W.decode_step_inputs, w, consts, s + 16)
            for key in kept:
                kept[key].append(x[key].reshape(NH, -1)[tidx].clone())
            d = {key: t.cuda() for key, t in x.items()}
            step = gdn.kda_recurrent_step if w.kind == "kda" else gdn.gdn_recurrent_step
            o = step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, scale=w.scale)
            outs.append(o.reshape(NH, w.dv)[tidx.cuda()].float().cpu())
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    # oracle: the sampled chains as independent sequences of T = steps tokens
    q, k, v = (torch.stack(kept[key], dim=1)[:, :, None] for key in ("q", "k", "v"))
    beta = torch.stack(kept["beta"], dim=1)[:, :, :1]
    g = torch.stack(kept["g"], dim=1)[:, :, None] if w.kind == "kda" else torch.stack(kept["g"], dim=1)[:, :, :1]
    o_ref, h_ref = oracle.recurrence(q, k, v, g, beta, w.scale, h0s, gate_per_channel=w.kind == "kda")
    o_gpu = torch.stack(outs, dim=1).double().numpy()
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    for s in range(steps):
        assert_close(o_gpu[:, s], o_ref[:, s, 0], dtype, f"o at step {s}")
    st = state.reshape(NH, w.dk, w.dv)[tidx.cuda()].double().cpu().numpy()
    assert_close(st, h_ref[:, 0], dtype, "state after the last step")


@pytest.mark.parametrize("N,H,dk,dv,dtype", [(3, 2, 16, 8, "f32"), (4, 2, 128, 128, "f32"), (5, 3, 128, 128, "bf16"),
                                             (2, 2, 64, 100, "bf16"), (3, 2, 256, 256, "bf16"), (2, 2, 256, 96, "f32")])
def test_small_decode(N, H, dk, dv, dtype):
    _decode_and_compare(W.DecodeWorkload("t", N, H, dk, dv, 40, dtype=dtype), 40)


@pytest.mark.parametrize("N,H,dk,dv,dtype", [(3, 2, 16, 8, "f32"), (4, 2, 128, 128, "f32"), (5, 3, 128, 128, "bf16"),
                                             (2, 2, 64, 100, "bf16"), (3, 2, 256, 256, "bf16")])
def test_small_kda_decode(N, H, dk, dv, dtype):
    _decode_and_compare(W.DecodeWorkload("t", N, H, dk, dv, 40, dtype=dtype, kind="kda"), 40)


def test_kda_decode_with_equal_channels_is_the_gdn_decode():
    w = W.DecodeWorkload("t", 6, 3, 128, 128, 1)
    c = W.decode_constants(w, seed=2)
    x = {k: v.cuda() for k, v in W.decode_step_inputs(w, c, 0).items()}
    s1, s2 = c["state"].cuda(), c["state"].cuda()
    o1 = gdn.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"], s1, scale=w.scale)
    gk = x["g"][..., None].expand(6, 3, 128).contiguous()
    o2 = gdn.kda_recurrent_step(x["q"], x["k"], x["v"], gk, x["beta"], s2, scale=w.scale)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_full_kda_decode_sampled_chains():
    w = W.DecodeWorkload("kda_decode", 256, 32, 128, 128, 64, kind="kda")
    _decode_and_compare(w, 64, sample=np.arange(0, 256 * 32, 97))


def test_bf16_output_is_the_rounded_fp32_output():
    w = W.DecodeWorkload("t", 8, 4, 128, 128, 1)
    c = W.decode_constants(w, seed=1)
    x = {k: v.cuda() for k, v in W.decode_step_inputs(w, c, 0).items()}
    s32, s16 = c["state"].cuda(), c["state"].cuda()
    o32 = gdn.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"], s32, scale=w.scale)
    o16 = gdn.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"], s16, scale=w.scale,
                                 o_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(s16, s32)


def test_full_decode_1024_steps_sampled_chains():
    w = W.config(4)
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(w.N * w.H, size=64, replace=False))
    _decode_and_compare(w, w.steps, sample=list(sample))


def test_decode_with_in_kernel_gate_and_beta_activation():
    w = W.DecodeWorkload("t", 8, 4, 128, 128, 24)
    consts = W.decode_constants(w, seed=3)
    rng = np.random.default_rng(3)
    A_log = np.log(rng.uniform(0.5, 16.0, size=w.H)).astype(np.float32)
    dt_bias = rng.normal(0.0, 0.1, size=w.H).astype(np.float32)
    state = consts["state"].cuda()
    NH = w.N * w.H
    qs, ks, vs, gs, bs, outs = [], [], [], [], [], []
    for s in range(w.steps):
        x = W.decode_step_inputs(w, consts, s)
        gl = rng.standard_normal((w.N, w.H), dtype=np.float32)
        bl = rng.standard_normal((w.N, w.H), dtype=np.float32)
        d = {k: v.cuda() for k, v in x.items()}
        o = gdn.gdn_recurrent_step(d["q"], d["k"], d["v"], torch.from_numpy(gl).cuda(), torch.from_numpy(bl).cuda(),
                                   state, scale=w.scale, A_log=torch.from_numpy(A_log).cuda(),
                                   dt_bias=torch.from_numpy(dt_bias).cuda(), beta_sigmoid=True)
        outs.append(o.reshape(NH, -1).float().cpu())
        qs.append(x["q"].reshape(NH, -1)); ks.append(x["k"].reshape(NH, -1)); vs.append(x["v"].reshape(NH, -1))
        gs.append(torch.from_numpy(oracle.gate_activation(gl, A_log, dt_bias)).reshape(NH, 1))
        bs.append(torch.from_numpy(oracle.beta_activation(bl)).reshape(NH, 1))
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    q, k, v = (torch.stack(t, dim=1)[:, :, None] for t in (qs, ks, vs))
    g, beta = torch.stack(gs, dim=1), torch.stack(bs, dim=1)
    o_ref, h_ref = oracle.recurrence(q, k, v, g, beta, w.scale, consts["state"].reshape(NH, 1, 128, 128))
    o_gpu = torch.stack(outs, dim=1).double().numpy()
    for s in range(w.steps):
        assert_close(o_gpu[:, s], o_ref[:, s, 0], torch.bfloat16, f"o at step {s}")
    assert_close(state.reshape(NH, 128, 128).double().cpu().numpy(), h_ref[:, 0], torch.bfloat16, "state")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_decode_grouped_value_heads(kind):
    Hk, G = 2, 4
    w = W.DecodeWorkload("t", 6, Hk * G, 128, 128, 12, kind=kind)
    consts = W.decode_constants(w, seed=4)
    state = consts["state"].cuda()
    NH = w.N * w.H
    qs, ks, vs, gs, bs, outs = [], [], [], [], [], []
    step = gdn.kda_recurrent_step if kind == "kda" else gdn.gdn_recurrent_step
    for s in range(w.steps):
        x = W.decode_step_inputs(w, consts, s)
        qk = {n: x[n][:, ::G].contiguous() for n in ("q", "k")}   # [N, Hk, d]
        d = {n: t.cuda() for n, t in x.items()}
        o = step(qk["q"].cuda(), qk["k"].cuda(), d["v"], d["g"], d["beta"], state, scale=w.scale)
        outs.append(o.reshape(NH, -1).float().cpu())
        qs.append(qk["q"].repeat_interleave(G, dim=1).reshape(NH, -1))
        ks.append(qk["k"].repeat_interleave(G, dim=1).reshape(NH, -1))
        vs.append(x["v"].reshape(NH, -1))
        gs.append(x["g"].reshape(NH, -1))
        bs.append(x["beta"].reshape(NH, 1))
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    q, k, v = (torch.stack(t, dim=1)[:, :, None] for t in (qs, ks, vs))
    beta = torch.stack(bs, dim=1)
    g = torch.stack(gs, dim=1)[:, :, None] if kind == "kda" else torch.stack(gs, dim=1)
    o_ref, h_ref = oracle.recurrence(q, k, v, g, beta, w.scale, consts["state"].reshape(NH, 1, 128, 128),
                                     gate_per_channel=kind == "kda")
    o_gpu = torch.stack(outs, dim=1).double().numpy()
    for s in range(w.steps):
        assert_close(o_gpu[:, s], o_ref[:, s, 0], torch.bfloat16, f"o at step {s}")
    assert_close(state.reshape(NH, 128, 128).double().cpu().numpy(), h_ref[:, 0], torch.bfloat16, "state")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_decode_beta_in_zero_two_from_logits(kind):
    w = W.DecodeWorkload("t", 5, 3, 128, 128, 16, kind=kind)
    consts = W.decode_constants(w, seed=5)
    rng = np.random.default_rng(5)
    state = consts["state"].cuda()
    NH = w.N * w.H
    step = gdn.kda_recurrent_step if kind == "kda" else gdn.gdn_recurrent_step
    qs, ks, vs, gs, bs, outs = [], [], [], [], [], []
    for s in range(w.steps):
        x = W.decode_step_inputs(w, consts, s)
        bl = rng.standard_normal((w.N, w.H), dtype=np.float32)
        d = {n: t.cuda() for n, t in x.items()}
        o = step(d["q"], d["k"], d["v"], d["g"], torch.from_numpy(bl).cuda(), state, scale=w.scale,
                 beta_sigmoid=True, allow_neg_eigval=True)
        outs.append(o.reshape(NH, -1).float().cpu())
        qs.append(x["q"].reshape(NH, -1)); ks.append(x["k"].reshape(NH, -1)); vs.append(x["v"].reshape(NH, -1))
        gs.append(x["g"].reshape(NH, -1))
        bs.append(torch.from_numpy(oracle.beta_activation(bl, 2)).reshape(NH, 1))
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    q, k, v = (torch.stack(t, dim=1)[:, :, None] for t in (qs, ks, vs))
    beta = torch.stack(bs, dim=1)
    g = torch.stack(gs, dim=1)[:, :, None] if kind == "kda" else torch.stack(gs, dim=1)
    o_ref, h_ref = oracle.recurrence(q, k, v, g, beta, w.scale, consts["state"].reshape(NH, 1, 128, 128),
                                     gate_per_channel=kind == "kda")
    o_gpu = torch.stack(outs, dim=1).double().numpy()
    for s in range(w.steps):
        assert_close(o_gpu[:, s], o_ref[:, s, 0], torch.bfloat16, f"o at step {s}")
    assert_close(state.reshape(NH, 128, 128).double().cpu().numpy(), h_ref[:, 0], torch.bfloat16, "state")

"""GPU parity of the chunk backward (gdn_chunk_bwd) against the fp64 oracle's backward.

Every call goes through the C ABI (ctypes binding) on seeded synthetic inputs
from gated_delta_rule_gdn_gb300.workloads, compared element by element with
oracle.recurrence_backward (itself pinned by finite differences of the forward
oracle):
* small cases the oracle runs whole: several chunks and a ragged tail, both gate
  forms, fp32 and bf16, chunk 16 and 32, partial and multi-tile d_v;
* the full-size workloads, on sampled (sequence, head) chains, which are
  independent, so the oracle runs on the chain alone;
* edge cases: packed sequences with an empty one, T < C, no initial state and no
  final-state gradient, beta up to 2, head sizes up to 256.
The result must not depend on scheduling (two runs are bitwise equal) nor on
whether the caller passes the workspace.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_gdn_gb300 as gdn
import oracle
from gated_delta_rule_gdn_gb300 import workloads as W
from parity_util import assert_close, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_gdn_gb300 import build
    build.build()
    gdn.load()


def _problem(kind, dtype, B, T, H, dk, dv, h0_std=0.5, dhT_std=1.0, seed=0, n_seqs=0, lens=None):
    w = W.ChunkWorkload("t", kind, B, T, H, dk, dv, 32, dtype, h0_std=h0_std)
    x = W.chunk_inputs(w, seed)
    if lens is not None:
        x["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
        x["N"] = len(lens)
        if h0_std > 0:
            rng = np.random.default_rng(seed + 7)
            x["initial_state"] = torch.from_numpy(
                (rng.standard_normal((len(lens), H, dk, dv)) * h0_std).astype(np.float32))
    x.update(W.chunk_output_grads(x, seed + 1, dhT_std))
    return x


def _gpu(x, chunk_size=0, workspace=None, want_dh0=True):
    d = to_dev(x)
    out = gdn.chunk_bwd(x["gate_per_channel"], d["q"], d["k"], d["v"], d["g"], d["beta"], d["d_o"],
                        scale=x["scale"], initial_state=d["initial_state"], d_final_state=d["d_final_state"],
                        cu_seqlens=d["cu_seqlens"], chunk_size=chunk_size, workspace=workspace,
                        want_d_initial_state=want_dh0)
    torch.cuda.synchronize()
    return {n: (None if t is None else t.double().cpu().numpy()) for n, t in zip(NAMES, out)}


def _oracle(x):
    return oracle.recurrence_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["d_o"],
                                      x["initial_state"], x["d_final_state"], cu_seqlens=x["cu_seqlens"],
                                      gate_per_channel=x["gate_per_channel"])


def _compare(got, ref, dtype, what, names=NAMES):
    for n in names:
        if got.get(n) is None:
            continue
        assert_close(got[n], ref[n], dtype, f"{what} {n}")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
@pytest.mark.parametrize("C", [16, 32])
def test_small_f32(kind, C):
    x = _problem(kind, "f32", 2, 100, 2, 64, 64)
    _compare(_gpu(x, C), _oracle(x), torch.float32, f"{kind} C{C}")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_small_bf16(kind):
    x = _problem(kind, "bf16", 2, 77, 2, 128, 128, h0_std=0.02)
    _compare(_gpu(x), _oracle(x), torch.bfloat16, kind)


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_packed_with_an_empty_sequence(kind):
    x = _problem(kind, "f32", 1, 0, 2, 32, 48, lens=[37, 0, 64, 1, 90])
    w = W.ChunkWorkload("t", kind, 1, 192, 2, 32, 48, 32, "f32", h0_std=0.0)
    y = W.chunk_inputs(w, 3)
    for n in ("q", "k", "v", "g", "beta"):
        x[n] = y[n]
    x.update(W.chunk_output_grads(x, 4))
    got = _gpu(x)
    _compare(got, _oracle(x), torch.float32, f"{kind} packed")
    # the empty sequence passes its final-state gradient through unchanged
    assert np.array_equal(got["dh0"][1], x["d_final_state"][1].double().numpy())


@pytest.mark.parametrize("kind,dk,dv", [("gdn", 24, 40), ("kda", 48, 16), ("gdn", 160, 96), ("kda", 64, 256),
                                        ("gdn", 256, 64), ("kda", 256, 32), ("gdn", 40, 37), ("kda", 33, 13)])
def test_head_sizes(kind, dk, dv):
    x = _problem(kind, "f32", 1, 45, 2, dk, dv, h0_std=0.3)
    _compare(_gpu(x), _oracle(x), torch.float32, f"{kind} dk{dk} dv{dv}")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_shorter_than_a_chunk_no_state_no_state_gradient(kind):
    x = _problem(kind, "f32", 3, 7, 1, 32, 32, h0_std=0.0, dhT_std=0.0)
    got = _gpu(x, want_dh0=False)
    assert got["dh0"] is None
    _compare(got, _oracle(x), torch.float32, kind, names=NAMES[:5])


def test_beta_up_to_two():
    x = _problem("gdn", "f32", 1, 96, 2, 64, 64)
    x["beta"] = 2.0 * x["beta"]
    _compare(_gpu(x), _oracle(x), torch.float32, "beta in (0, 2)")


def test_bitwise_repeatable_and_workspace_independent():
    x = _problem("kda", "bf16", 2, 130, 3, 64, 96, h0_std=0.02)
    a = _gpu(x)
    need = gdn.bwd_workspace_size(True, 2, 130, 3, 64, 96)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    b = _gpu(x, workspace=ws)
    for n in NAMES:
        assert np.array_equal(a[n], b[n]), n


def test_chunk_size_sets_rounding_only():
    x = _problem("gdn", "f32", 1, 200, 2, 64, 64)
    a, b = _gpu(x, 16), _gpu(x, 32)
    for n in NAMES:
        assert_close(a[n], b[n], torch.float32, f"C16 vs C32 {n}")


# --- full-size workloads, sampled chains -----------------------------------------------------------

def _chain(x, b, h):
    """The inputs of one (batch row, head) chain, as a problem of its own."""
    y = {"scale": x["scale"], "gate_per_channel": x["gate_per_channel"], "cu_seqlens": None, "N": 1}
    for n in ("q", "k", "v", "g", "beta", "d_o"):
        y[n] = x[n][b:b + 1, :, h:h + 1]
    for n in ("initial_state", "d_final_state"):
        y[n] = None if x[n] is None else x[n][b:b + 1, h:h + 1]
    return y


@pytest.mark.parametrize("cfg,chains", [(1, [(0, 3), (3, 15)]), (3, [(1, 30)])])
def test_full_size_sampled_chains(cfg, chains):
    w = W.config(cfg)
    x = W.chunk_inputs(w, 0)
    x.update(W.chunk_output_grads(x, 1, dhT_std=0.02))
    got = _gpu(x)
    for b, h in chains:
        y = _chain(x, b, h)
        ref = _oracle(y)
        sub = {n: (got[n][b:b + 1, :, h:h + 1] if n != "dh0" else got[n][b:b + 1, h:h + 1]) for n in NAMES}
        _compare(sub, ref, x["q"].dtype, f"config {cfg} chain ({b}, {h})")


def test_full_size_packed_sampled_chains():
    w = W.config(2)
    x = W.chunk_inputs(w, 0)
    x.update(W.chunk_output_grads(x, 1, dhT_std=0.02))
    got = _gpu(x)
    cu = x["cu_seqlens"].numpy()
    for n, h in ((0, 5), (5, 31)):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        y = {"scale": x["scale"], "gate_per_channel": False, "cu_seqlens": None, "N": 1}
        for m in ("q", "k", "v", "g", "beta", "d_o"):
            y[m] = x[m][:, t0:t1, h:h + 1]
        y["initial_state"] = x["initial_state"][n:n + 1, h:h + 1]
        y["d_final_state"] = x["d_final_state"][n:n + 1, h:h + 1]
        ref = _oracle(y)
        sub = {m: (got[m][:, t0:t1, h:h + 1] if m != "dh0" else got[m][n:n + 1, h:h + 1]) for m in NAMES}
        _compare(sub, ref, x["q"].dtype, f"packed sequence {n} head {h}")


def test_a_walk_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    # the test injection leaves out the first chunk record's copy: the walks' bounded wait gives up (about 2 s)
    x = _problem("gdn", "bf16", 1, 64, 2, 128, 128, h0_std=0.02)
    lib = gdn.load()
    gdn.device_status()                       # start from a clear status
    assert lib.gdn_test_inject(1) == 0
    _gpu(x)                                   # this call's gradients are unspecified
    assert gdn.device_status() == 4           # GDN_ERR_TIMEOUT, and cleared
    assert gdn.device_status() == 0
    _compare(_gpu(x), _oracle(x), torch.bfloat16, "after the timeout")
    assert gdn.device_status() == 0


@pytest.mark.parametrize("kind,mult", [("gdn", 1), ("gdn", 2), ("kda", 1), ("kda", 2)])
def test_activations_in_the_path(kind, mult):
    # g and beta as raw logits: log alpha = -exp(A_log) softplus(g + dt_bias) (scalar gate), beta = mult sigmoid(b);
    # the oracle composes its activation, its backward and the activation's chain rule
    x = _problem(kind, "bf16", 2, 100, 2, 64, 64, h0_std=0.02)
    rng = np.random.default_rng(21)
    B, T, H = x["beta"].shape
    b_raw = rng.standard_normal((B, T, H)).astype(np.float32)
    kw = dict(beta_sigmoid=True, allow_neg_eigval=mult == 2)
    if kind == "gdn":
        g_raw = rng.standard_normal((B, T, H)).astype(np.float32)
        A_log = np.log(rng.uniform(0.5, 16.0, H)).astype(np.float32)
        dt = rng.normal(0.0, 0.1, H).astype(np.float32)
        g64 = oracle.gate_activation(g_raw, A_log, dt)
        kw.update(A_log=torch.from_numpy(A_log).cuda(), dt_bias=torch.from_numpy(dt).cuda())
    else:
        g_raw, A_log, dt = x["g"].numpy(), None, None
        g64 = g_raw
    y = dict(x)
    y["g"], y["beta"] = g64, oracle.beta_activation(b_raw, mult)
    ref = _oracle(y)
    ch = oracle.activation_backward(g_raw, b_raw, A_log, dt, mult, ref["dg"], ref["dbeta"])
    d = to_dev(x)
    out = gdn.chunk_bwd(kind == "kda", d["q"], d["k"], d["v"], torch.from_numpy(g_raw).cuda(),
                        torch.from_numpy(b_raw).cuda(), d["d_o"], scale=x["scale"], initial_state=d["initial_state"],
                        d_final_state=d["d_final_state"], **kw)
    torch.cuda.synchronize()
    got = [None if t is None else t.double().cpu().numpy() for t in out]
    for n, i in (("dq", 0), ("dk", 1), ("dv", 2), ("dh0", 5)):
        assert_close(got[i], ref[n], torch.bfloat16, f"{kind} act {n}")
    assert_close(got[3], ch["dx"], torch.bfloat16, f"{kind} act d(gate logit)")
    assert_close(got[4], ch["db"], torch.bfloat16, f"{kind} act d(beta logit)")
    if kind == "gdn":
        assert_close(got[6], ch["dA_log"], torch.float32, "dA_log")
        assert_close(got[7], ch["ddt_bias"], torch.float32, "ddt_bias")
    else:
        assert got[6] is None and got[7] is None


@pytest.mark.parametrize("kind,dtype", [("gdn", "f32"), ("kda", "f32"), ("gdn", "bf16")])
def test_grouped_value_heads(kind, dtype):
    # H_v = 3 H_k: value head h reads q, k of key head h // 3; the oracle runs on q, k repeated per value head and
    # the gradient of a shared key head is the sum over its value heads
    Hk, G = 2, 3
    x = _problem(kind, dtype, 2, 70, Hk * G, 64, 48, h0_std=0.3 if dtype == "f32" else 0.02)
    qk = {n: x[n][:, :, :Hk].contiguous() for n in ("q", "k")}
    y = dict(x)
    for n in ("q", "k"):
        y[n] = qk[n].repeat_interleave(G, dim=2)
    ref = _oracle(y)
    d = to_dev(x)
    out = gdn.chunk_bwd(kind == "kda", qk["q"].cuda(), qk["k"].cuda(), d["v"], d["g"], d["beta"], d["d_o"],
                        scale=x["scale"], initial_state=d["initial_state"], d_final_state=d["d_final_state"])
    torch.cuda.synchronize()
    got = [t.double().cpu().numpy() for t in out]
    B, T = x["q"].shape[:2]
    tol = torch.float32 if dtype == "f32" else torch.bfloat16
    assert got[0].shape == (B, T, Hk, 64)
    assert_close(got[0], ref["dq"].reshape(B, T, Hk, G, 64).sum(3), tol, f"{kind} GVA dq")
    assert_close(got[1], ref["dk"].reshape(B, T, Hk, G, 64).sum(3), tol, f"{kind} GVA dk")
    for n, i in (("dv", 2), ("dg", 3), ("dbeta", 4), ("dh0", 5)):
        assert_close(got[i], ref[n], tol, f"{kind} GVA {n}")


def test_grouped_value_heads_with_activations():
    # both at once: q, k of key head h // 2 serve value heads h; g and beta are raw logits activated in the path
    Hk, G = 2, 2
    x = _problem("gdn", "bf16", 2, 90, Hk * G, 64, 48, h0_std=0.02)
    rng = np.random.default_rng(23)
    B, T, H = x["beta"].shape
    g_raw = rng.standard_normal((B, T, H)).astype(np.float32)
    b_raw = rng.standard_normal((B, T, H)).astype(np.float32)
    A_log = np.log(rng.uniform(0.5, 16.0, H)).astype(np.float32)
    dt = rng.normal(0.0, 0.1, H).astype(np.float32)
    qk = {n: x[n][:, :, :Hk].contiguous() for n in ("q", "k")}
    y = dict(x)
    for n in ("q", "k"):
        y[n] = qk[n].repeat_interleave(G, dim=2)
    y["g"], y["beta"] = oracle.gate_activation(g_raw, A_log, dt), oracle.beta_activation(b_raw, 1)
    ref = _oracle(y)
    ch = oracle.activation_backward(g_raw, b_raw, A_log, dt, 1, ref["dg"], ref["dbeta"])
    d = to_dev(x)
    out = gdn.chunk_bwd(False, qk["q"].cuda(), qk["k"].cuda(), d["v"], torch.from_numpy(g_raw).cuda(),
                        torch.from_numpy(b_raw).cuda(), d["d_o"], scale=x["scale"], initial_state=d["initial_state"],
                        d_final_state=d["d_final_state"], A_log=torch.from_numpy(A_log).cuda(),
                        dt_bias=torch.from_numpy(dt).cuda(), beta_sigmoid=True)
    torch.cuda.synchronize()
    got = [t.double().cpu().numpy() for t in out]
    assert_close(got[0], ref["dq"].reshape(B, T, Hk, G, 64).sum(3), torch.bfloat16, "GVA act dq")
    assert_close(got[1], ref["dk"].reshape(B, T, Hk, G, 64).sum(3), torch.bfloat16, "GVA act dk")
    assert_close(got[2], ref["dv"], torch.bfloat16, "GVA act dv")
    assert_close(got[5], ref["dh0"], torch.bfloat16, "GVA act dh0")
    assert_close(got[3], ch["dx"], torch.bfloat16, "GVA act d(gate logit)")
    assert_close(got[4], ch["db"], torch.bfloat16, "GVA act d(beta logit)")
    assert_close(got[6], ch["dA_log"], torch.float32, "GVA act dA_log")
    assert_close(got[7], ch["ddt_bias"], torch.float32, "GVA act ddt_bias")

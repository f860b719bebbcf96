"""Pins for the oracle's backward (oracle.recurrence_backward).

The gradients of L = <dO, o> + <dhT, h_final> are fixed by the forward
recurrence, so the backward is pinned to the forward oracle (itself pinned in
test_oracle_pins.py) by central finite differences in random directions, one
check per input.  This check shares no code with the adjoint.  Closed forms add
exact checks:
* at beta = 0 the state is the decayed entry state, so dk = dv = 0 and dq has a
  closed form;
* packed sequences give the gradients of separate runs, bit for bit.
Planted slips in a copy of the adjoint must fail these checks.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")


def _case(seed, B=2, T=11, H=2, dk=5, dv=4, kda=False, h0=True, beta_hi=0.95):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk)) / np.sqrt(dk)
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, beta_hi, (B, T, H))
    g = -rng.uniform(0.0, 0.6, (B, T, H, dk) if kda else (B, T, H))
    S0 = rng.standard_normal((B, H, dk, dv)) if h0 else None
    dO = rng.standard_normal((B, T, H, dv))
    dhT = rng.standard_normal((B, H, dk, dv))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, dO=dO, dhT=dhT)


def _loss(c, scale, cu=None):
    o, hT = oracle.recurrence(c["q"], c["k"], c["v"], c["g"], c["beta"], scale, c["S0"], cu_seqlens=cu)
    return float(np.sum(o * c["dO"]) + np.sum(hT * c["dhT"]))


def _grads(c, scale, cu=None):
    return oracle.recurrence_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], scale, c["dO"], c["S0"],
                                      c["dhT"], cu_seqlens=cu)


NAMES = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "S0": "dh0"}


def _fd_errors(c, scale, grads, cu=None, seed=99, eps=1e-6):
    """Relative error of <grad, E> against (L(x + eps E) - L(x - eps E)) / (2 eps), per input."""
    rng = np.random.default_rng(seed)
    errs = {}
    for name, gname in NAMES.items():
        if c[name] is None:
            continue
        E = rng.standard_normal(c[name].shape)
        cp = dict(c); cp[name] = c[name] + eps * E
        cm = dict(c); cm[name] = c[name] - eps * E
        fd = (_loss(cp, scale, cu) - _loss(cm, scale, cu)) / (2 * eps)
        an = float(np.sum(grads[gname] * E))
        errs[name] = abs(fd - an) / max(abs(fd), 1e-3)
    return errs


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_gradients_match_central_differences(seed, kda):
    c = _case(seed, kda=kda)
    errs = _fd_errors(c, 0.8, _grads(c, 0.8))
    assert max(errs.values()) < 1e-6, errs


def test_gradients_match_central_differences_beta_up_to_two():
    # beta in (0, 2): the negative-eigenvalue range; the same gradient formulas hold
    c = _case(2, beta_hi=1.95)
    errs = _fd_errors(c, 1.1, _grads(c, 1.1))
    assert max(errs.values()) < 1e-6, errs


def test_gradients_packed_sequences_central_differences():
    c = _case(3, B=1, T=17, H=2)
    cu = np.array([0, 5, 5, 12, 17], dtype=np.int32)
    rng = np.random.default_rng(4)
    c["S0"] = rng.standard_normal((4, 2, 5, 4))
    c["dhT"] = rng.standard_normal((4, 2, 5, 4))
    errs = _fd_errors(c, 0.8, _grads(c, 0.8, cu), cu=cu)
    assert max(errs.values()) < 1e-6, errs


def test_beta_zero_closed_form():
    # beta = 0: h_t = exp(g_1 + ... + g_t) h0, nothing depends on k or v
    c = _case(5)
    c["beta"] = np.zeros_like(c["beta"])
    scale = 0.7
    gr = _grads(c, scale)
    assert np.all(gr["dk"] == 0.0) and np.all(gr["dv"] == 0.0)
    cum = np.exp(np.cumsum(c["g"], axis=1))                       # [B, T, H]
    ht = cum[..., None, None] * c["S0"][:, None]                  # [B, T, H, dk, dv]
    dq = scale * np.einsum("bthij,bthj->bthi", ht, c["dO"])
    assert np.max(np.abs(gr["dq"] - dq)) < 1e-13
    # dh0 = sum_t scale exp(G_t) q_t dO_t^T + exp(G_T) dhT
    dh0 = scale * np.einsum("bth,bthi,bthj->bhij", cum, c["q"], c["dO"]) + cum[:, -1][..., None, None] * c["dhT"]
    assert np.max(np.abs(gr["dh0"] - dh0)) < 1e-12


def test_packed_gradients_equal_separate_runs_bitwise():
    c = _case(6, B=1, T=14, H=2)
    cu = np.array([0, 6, 14], dtype=np.int32)
    rng = np.random.default_rng(7)
    c["S0"] = rng.standard_normal((2, 2, 5, 4))
    c["dhT"] = rng.standard_normal((2, 2, 5, 4))
    gp = _grads(c, 0.9, cu)
    for n in range(2):
        a, b = cu[n], cu[n + 1]
        cs = {key: (val[:, a:b] if key in ("q", "k", "v", "g", "beta", "dO") else val[n:n + 1])
              for key, val in c.items()}
        gs = _grads(cs, 0.9)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            assert np.array_equal(gp[key][:, a:b], gs[key]), key
        assert np.array_equal(gp["dh0"][n:n + 1], gs["dh0"])


def test_zero_length_sequence_passes_the_state_gradient_through():
    c = _case(8, B=1, T=4, H=1)
    cu = np.array([0, 0, 4], dtype=np.int32)
    rng = np.random.default_rng(9)
    c["S0"] = rng.standard_normal((2, 1, 5, 4))
    c["dhT"] = rng.standard_normal((2, 1, 5, 4))
    gr = _grads(c, 0.8, cu)
    assert np.array_equal(gr["dh0"][0], c["dhT"][0])


# --- planted slips in a copy of the adjoint --------------------------------------------

MUTATIONS = {
    "dk_drops_state_term": ("kd += G[i * dv + j] * r[j] + a[i * dv + j] * dp[j];",
                            "kd += G[i * dv + j] * r[j];"),
    "dp_sign": ("dp[j] = -bt * dr[j];", "dp[j] = bt * dr[j];"),
    "state_gradient_not_decayed": ("G[i * dv + j] = al[i] * dai;", "G[i * dv + j] = dai;"),
    "dg_without_alpha": ("if (gate_per_channel) dg[tok * dk + i] = al[i] * sa;",
                         "if (gate_per_channel) dg[tok * dk + i] = sa;"),
    "dq_reads_entry_state": ("sq += hn[i * dv + j] * dot[j];", "sq += hp[i * dv + j] * dot[j];"),
    "dbeta_uses_value": ("db += dr[j] * (vt[j] - p[j]);", "db += dr[j] * vt[j];"),
    "read_gradient_after_write_backprop": (
        "                G[i * dv + j] += scale * qt[i] * dot[j];\n", ""),
}


def _load_mutant(old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = os.path.join(tmp, "mut.c")
    open(path, "w").write(src.replace(old, new))
    lib = os.path.join(tmp, "libmut.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", "-o", lib, path, "-lm"],
                   check=True)
    return lib


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_backward_mutation(name, monkeypatch):
    real = oracle.load()
    with tempfile.TemporaryDirectory() as tmp:
        lib = ctypes.CDLL(_load_mutant(*MUTATIONS[name], tmp))
        lib.gdn_oracle_backward.restype = ctypes.c_int
        lib.gdn_oracle_backward.argtypes = real.gdn_oracle_backward.argtypes
        lib.gdn_oracle_forward.restype = ctypes.c_int
        lib.gdn_oracle_forward.argtypes = real.gdn_oracle_forward.argtypes
        monkeypatch.setattr(oracle, "_lib", lib)
        caught = False
        for kda in (False, True):
            c = _case(10, kda=kda)
            errs = _fd_errors(c, 0.8, _grads(c, 0.8))
            if max(errs.values()) > 1e-4:
                caught = True
        assert caught, name


# --- the activations around the backward -----------------------------------------------------------------

@pytest.mark.parametrize("mult", [1, 2])
def test_activation_chain_rule_matches_central_differences(mult):
    # L(x, b, A_log, dt_bias) = <dO, o> + <dhT, h_T> with log alpha and beta formed from raw logits
    c = _case(11, T=9)
    rng = np.random.default_rng(12)
    B, T, H = c["beta"].shape
    x = rng.standard_normal((B, T, H))
    b = rng.standard_normal((B, T, H))
    A_log = np.log(rng.uniform(0.5, 4.0, H))
    dt = rng.normal(0.0, 0.3, H)
    scale = 0.8

    def loss(x_, b_, A_, dt_):
        d = dict(c)
        d["g"] = oracle.gate_activation(x_, A_, dt_)
        d["beta"] = oracle.beta_activation(b_, mult)
        return _loss(d, scale)

    d = dict(c)
    d["g"] = oracle.gate_activation(x, A_log, dt)
    d["beta"] = oracle.beta_activation(b, mult)
    gr = _grads(d, scale)
    ch = oracle.activation_backward(x, b, A_log, dt, mult, gr["dg"], gr["dbeta"])
    eps = 1e-6
    args = [x, b, A_log, dt]
    names = ["dx", "db", "dA_log", "ddt_bias"]
    for i, name in enumerate(names):
        E = rng.standard_normal(args[i].shape)
        ap = list(args); ap[i] = args[i] + eps * E
        am = list(args); am[i] = args[i] - eps * E
        fd = (loss(*ap) - loss(*am)) / (2 * eps)
        an = float(np.sum(ch[name] * E))
        assert abs(fd - an) <= 1e-6 * max(abs(fd), 1e-3), (name, fd, an)


def test_activations_match_their_definitions_at_known_points():
    # softplus(0) = log 2, sigmoid(0) = 1/2; beta doubles with mult 2
    assert np.isclose(oracle.gate_activation(np.zeros(1), np.zeros(1), None)[0], -np.log(2.0), rtol=0, atol=1e-15)
    assert np.isclose(oracle.beta_activation(np.zeros(1), 2)[0], 1.0, rtol=0, atol=1e-15)
    assert np.isclose(oracle.gate_activation(np.array([30.0]), np.array([np.log(3.0)]), np.array([1.0]))[0], -93.0,
                      rtol=1e-12)

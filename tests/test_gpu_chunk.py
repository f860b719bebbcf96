"""GPU parity of the chunk forward (gdn_chunk_fwd, kda_chunk_fwd) against the fp64 oracle.

Every call goes through the C ABI (ctypes binding), on seeded synthetic inputs
from gated_delta_rule_gdn_gb300.workloads, in element-by-element comparison:
* small cases the oracle runs whole, spanning several chunks and a ragged tail;
* the full-size workloads (configs 1, 2 and 3, and the head-size-256 prefill), with the oracle run on every head;
* head size 256 on its tensor-core pair: ragged, packed, grouped value heads, in-kernel activations;
* edge cases: T < C, T = 0, zero-length packed sequences, extreme decay, beta
  near 0 and 1.
Packed sequences must match separate runs bitwise; so must a state hand-off at
a chunk boundary.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_gdn_gb300 as gdn
import oracle
from gated_delta_rule_gdn_gb300 import workloads as W
from parity_util import assert_close, oracle_on_heads, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_gdn_gb300 import build
    build.build()
    gdn.load()


def _fits(x, algo):
    """True if the library's kernel `algo` accepts this problem (asked through gdn_chunk_plan)."""
    B, T, H, dk = x["q"].shape
    try:
        gdn.chunk_plan(x["gate_per_channel"], B, T, H, dk, x["v"].shape[-1], x["chunk_size"], x["q"].dtype,
                       x["cu_seqlens"] is not None, algo)
        return True
    except gdn.GdnError:
        return False


def _run(x, algo="auto", out_final=True, o_dtype=torch.float32, workspace=None):
    d = to_dev(x)
    fn = gdn.kda_chunk_fwd if x["gate_per_channel"] else gdn.gdn_chunk_fwd
    o, hT = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["initial_state"],
               output_final_state=out_final, cu_seqlens=d["cu_seqlens"], chunk_size=x["chunk_size"], algo=algo,
               o_dtype=o_dtype, workspace=workspace)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    return o.double().cpu().numpy(), (None if hT is None else hT.double().cpu().numpy())


def _algos(x):
    return ["generic"] + [a for a in ("two_pass",) if _fits(x, a)]


def _workload(kind, dtype, dk, dv, C, h0_std):
    return W.ChunkWorkload("t", kind, 1, 1, 1, dk, dv, C, dtype, h0_std=h0_std)


def test_config0_tiny_fp32():
    x = W.chunk_inputs(W.config(0), seed=0)
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "auto")
    assert_close(o, o_ref, torch.float32, "o")
    assert_close(hT, h_ref, torch.float32, "final state")


SMALL = [
    # kind, dtype, B, T, H, dk, dv, C, h0
    ("gdn", "f32", 2, 200, 2, 32, 48, 64, 0.1),
    ("gdn", "f32", 1, 77, 3, 16, 16, 16, 0.0),
    ("gdn", "bf16", 2, 333, 2, 128, 128, 64, 0.02),
    ("gdn", "bf16", 1, 64, 2, 128, 128, 64, 0.02),
    ("gdn", "bf16", 3, 5, 2, 128, 128, 64, 0.02),
    ("gdn", "bf16", 1, 1, 1, 128, 128, 64, 0.02),
    ("gdn", "bf16", 2, 130, 2, 64, 96, 32, 0.05),
    ("gdn", "bf16", 1, 100, 2, 100, 72, 16, 0.0),
    ("kda", "f32", 1, 150, 2, 32, 32, 32, 0.1),
    ("kda", "bf16", 2, 200, 2, 128, 128, 64, 0.02),
    ("kda", "bf16", 1, 70, 2, 64, 128, 16, 0.0),
    ("gdn", "f32", 1, 90, 2, 40, 37, 16, 0.1),
    ("kda", "bf16", 1, 50, 2, 33, 13, 32, 0.0),
    # head sizes above 128 (the generic kernel; the per-channel gate at d_k = 256 takes chunk <= 32)
    ("gdn", "bf16", 2, 150, 2, 256, 256, 64, 0.02),
    ("gdn", "f32", 1, 90, 2, 256, 96, 32, 0.05),
    ("gdn", "bf16", 1, 70, 1, 160, 200, 16, 0.0),
    ("kda", "bf16", 1, 100, 2, 256, 256, 32, 0.02),
    ("kda", "f32", 1, 45, 1, 192, 256, 16, 0.0),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_small_shapes(case):
    kind, dt, B, T, H, dk, dv, C, h0 = case
    x = W.chunk_inputs(_workload(kind, dt, dk, dv, C, h0), seed=1, B=B, T=T, H=H)
    dtype = x["q"].dtype
    o_ref, h_ref = oracle_on_heads(x)
    for algo in _algos(x):
        o, hT = _run(x, algo)
        assert_close(o, o_ref, dtype, f"o [{algo}]")
        assert_close(hT, h_ref, dtype, f"final state [{algo}]")


def test_extreme_gates_and_betas():
    # A up to 16 drives gamma^r to 0 within a chunk (a correct underflow, never NaN); beta near 0 and 1
    x = W.chunk_inputs(W.config(1), seed=2, B=1, T=256, H=4)
    x["g"] = torch.clamp(x["g"] * 4.0, min=-80.0)
    x["beta"][..., 0] = 1e-6
    x["beta"][..., 1] = 1.0 - 1e-6
    o_ref, h_ref = oracle_on_heads(x)
    for algo in _algos(x):
        o, hT = _run(x, algo)
        assert_close(o, o_ref, torch.bfloat16, f"o [{algo}]")
        assert_close(hT, h_ref, torch.bfloat16, f"final state [{algo}]")


def test_kda_strong_per_channel_decay():
    """Per-channel decays far beyond what the factored intra-chunk products take (the kernel then forms every
    term with its own exponential), next to channels with mild decay, and chunks where only some blocks decay."""
    x = W.chunk_inputs(W.config(3), seed=4, B=1, T=200, H=2)
    g = x["g"].clone()
    g[:, :, 0, :16] = -30.0                 # head 0: 16 channels lose everything within a block
    g[:, 64:80, 1, 5] = -12.0               # head 1: one channel, one block of one chunk
    x["g"] = g
    o_ref, h_ref = oracle_on_heads(x)
    for algo in _algos(x):
        o, hT = _run(x, algo)
        assert_close(o, o_ref, torch.bfloat16, f"o [{algo}]")
        assert_close(hT, h_ref, torch.bfloat16, f"final state [{algo}]")


def test_kda_several_chunks_per_cta():
    """Enough chunks that every CTA of the per-chunk kernel walks several of them (loads of the next chunk overlap
    the current one)."""
    x = W.chunk_inputs(W.config(3), seed=6, B=1, T=4096 + 37, H=8)
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "auto")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_more_chains_than_sms(kind):
    """More (sequence, head, d_v half) chains than SMs in a uniform batch: the state pass runs in several waves."""
    x = W.chunk_inputs(W.config(3 if kind == "kda" else 1), seed=8, B=3, T=150, H=30)
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "auto")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_short_chains_in_a_deep_grid(kind):
    """384 short chains (768 state CTAs, five waves on 152 SMs) and 3,072 per-chunk items."""
    x = W.chunk_inputs(_workload(kind, "bf16", 128, 128, 64, 0.02), seed=11, B=8, T=256, H=48)
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "two_pass")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


def test_packed_long_and_short_sequences_in_a_deep_grid():
    """One long sequence among short and empty ones, 64 heads (several waves of state CTAs, longest first): parity,
    the empty sequence keeps its initial state, and a sequence's outputs do not depend on another's inputs."""
    lens = [1500, 64, 100, 37, 0, 300, 129]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    H = 64
    x = W.chunk_inputs(_workload("gdn", "bf16", 128, 128, 64, 0.02), seed=12, B=1, T=int(cu[-1]), H=H)
    x["cu_seqlens"] = torch.from_numpy(cu)
    x["initial_state"] = torch.randn(len(lens), H, 128, 128, generator=torch.Generator().manual_seed(1)) * 0.02
    o, hT = _run(x, "two_pass")
    o_ref, h_ref = oracle_on_heads(x)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")
    assert np.array_equal(hT[4], x["initial_state"][4].double().numpy())
    x2 = {**x, "v": x["v"].clone()}
    x2["v"][:, cu[5]:cu[6]] += 1.0
    o2, h2 = _run(x2, "two_pass")
    keep = np.ones(int(cu[-1]), bool)
    keep[cu[5]:cu[6]] = False
    assert np.array_equal(o2[:, keep], o[:, keep]) and np.array_equal(np.delete(h2, 5, 0), np.delete(hT, 5, 0))


def test_zero_length_input_keeps_initial_state():
    x = W.chunk_inputs(W.config(1), seed=3, B=2, T=0, H=2)
    for algo in _algos(x):
        o, hT = _run(x, algo)
        assert o.shape == (2, 0, 2, 128)
        assert np.array_equal(hT, x["initial_state"].double().numpy())


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_packed_sequences_match_separate_runs_bitwise(kind):
    lens = [130, 0, 64, 1, 200, 63, 65]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = W.chunk_inputs(_workload(kind, "bf16", 128, 128, 64, 0.02), seed=4, B=1, T=int(cu[-1]), H=3)
    x["cu_seqlens"] = torch.from_numpy(cu)
    x["initial_state"] = torch.randn(len(lens), 3, 128, 128, generator=torch.Generator().manual_seed(0)) * 0.02
    for algo in _algos(x):
        o, hT = _run(x, algo)
        for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
            xn = {**x, "cu_seqlens": None, "initial_state": x["initial_state"][n:n + 1]}
            for key in ("q", "k", "v", "g", "beta"):
                xn[key] = x[key][:, a:b].contiguous()
            on, hn = _run(xn, algo)
            assert np.array_equal(o[:, a:b], on), (algo, n)
            assert np.array_equal(hT[n], hn[0]), (algo, n)
        # perturbing one sequence leaves every other sequence's outputs bitwise unchanged
        x2 = {**x, "v": x["v"].clone()}
        x2["v"][:, cu[4]:cu[5]] += 1.0
        o2, h2 = _run(x2, algo)
        keep = np.ones(int(cu[-1]), bool)
        keep[cu[4]:cu[5]] = False
        assert np.array_equal(o2[:, keep], o[:, keep]) and np.array_equal(np.delete(h2, 4, 0), np.delete(hT, 4, 0))
        o_ref, h_ref = oracle_on_heads(x)
        assert_close(o, o_ref, torch.bfloat16, f"o [{algo}]")
        assert_close(hT, h_ref, torch.bfloat16, f"final state [{algo}]")


def test_state_handoff_at_chunk_boundary_is_bitwise():
    x = W.chunk_inputs(W.config(1), seed=5, B=1, T=320, H=2)
    for algo in _algos(x):
        o, hT = _run(x, algo)
        T1 = 192
        xa = {**x}
        xb = {**x}
        for key in ("q", "k", "v", "g", "beta"):
            xa[key] = x[key][:, :T1].contiguous()
            xb[key] = x[key][:, T1:].contiguous()
        oa, ha = _run(xa, algo)
        xb["initial_state"] = torch.from_numpy(ha).float()
        ob, hb = _run(xb, algo)
        assert np.array_equal(np.concatenate([oa, ob], axis=1), o) and np.array_equal(hb, hT)


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_bf16_output_is_the_rounded_fp32_output(kind):
    # a bf16 o is the round-to-nearest-even of the same fp32 result, bit for bit
    x = W.chunk_inputs(_workload(kind, "bf16", 128, 128, 64, 0.02), seed=7, B=2, T=150, H=2)
    for algo in _algos(x):
        o32, h32 = _run(x, algo)
        o16, h16 = _run(x, algo, o_dtype=torch.bfloat16)
        expect = torch.from_numpy(o32).float().to(torch.bfloat16).double().numpy()
        assert np.array_equal(o16, expect) and np.array_equal(h16, h32)


def test_kda_with_equal_channels_matches_gdn():
    x = W.chunk_inputs(W.config(1), seed=6, B=1, T=200, H=2)
    xk = {**x, "g": x["g"][..., None].expand(*x["g"].shape, 128).contiguous(), "gate_per_channel": True}
    og, hg = _run(x, "generic")
    ok, hk = _run(xk, "generic")
    assert_close(ok, og, torch.bfloat16, "o")
    assert_close(hk, hg, torch.bfloat16, "final state")


# --- full-size workloads, in the launch configuration the benchmark times -------------------

def test_benchmark_workload_runs_a_tensor_core_kernel():
    w = W.config(1)
    assert gdn.chunk_plan(False, w.B, w.T, w.H, w.dk, w.dv, w.chunk_size, torch.bfloat16) == "two_pass"


@pytest.mark.parametrize("algo", ["auto"])
def test_full_config1_all_chains(algo):
    x = W.chunk_inputs(W.config(1), seed=0)
    o_ref, h_ref = _oracle_cached(1, x)
    o, hT = _run(x, algo)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


@pytest.mark.parametrize("algo", ["auto"])
def test_full_config2_varlen_all_heads(algo):
    x = W.chunk_inputs(W.config(2), seed=0)
    o_ref, h_ref = _oracle_cached(2, x)
    o, hT = _run(x, algo)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


_ORACLE = {}


def _oracle_cached(key, x, heads=None):
    if key not in _ORACLE:
        _ORACLE[key] = oracle_on_heads(x, heads)
    return _ORACLE[key]


def test_two_pass_workspace_reuse_and_library_allocation():
    """A caller workspace reused across calls, and the library's own stream-ordered allocation (C entry
    point without a workspace), give bitwise the same result."""
    x = W.chunk_inputs(W.config(1), seed=3, T=700, H=3)
    B, T, H, dk = x["q"].shape
    n = gdn.workspace_size(False, B, T, H, dk, dk, 64, torch.bfloat16, 0, "two_pass")
    assert n == (B * T // 64 + B + 1) * H * 32768
    ws = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    o1, h1 = _run(x, "two_pass", workspace=ws)
    o2, h2 = _run(x, "two_pass", workspace=ws)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)
    o3, h3 = _run_c_entry(x, "two_pass")
    assert np.array_equal(o1, o3) and np.array_equal(h1, h3)
    with pytest.raises(gdn.GdnError):
        _run(x, "two_pass", workspace=ws[: n - 256])


def _run_c_entry(x, algo):
    """gdn_chunk_fwd_algo straight through ctypes: no workspace argument, so the library allocates one."""
    import ctypes
    lib = gdn.load()
    d = to_dev(x)
    B, T, H, dk = x["q"].shape
    o = torch.empty((B, T, H, dk), dtype=torch.float32, device="cuda")
    hT = torch.empty_like(d["initial_state"])
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.gdn_chunk_fwd_algo(p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]), p(d["beta"]), float(x["scale"]),
                                p(d["initial_state"]), 1, p(hT), None, 0, p(o), B, T, H, dk, dk, 64, 1, 0,
                                gdn._binding.ALGOS[algo], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, gdn.last_error()
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    return o.double().cpu().numpy(), hT.double().cpu().numpy()


def test_full_config3_kda_all_heads():
    x = W.chunk_inputs(W.config(3), seed=0)
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "auto")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


@pytest.mark.parametrize("algo", ["auto", "generic"])
def test_full_head256_all_heads(algo):
    # head size 256 at full size (B4 T4096 H8): the tensor-core pair (the launch the bench times) and the generic
    # kernel
    x = W.chunk_inputs(W.HEAD256, seed=0)
    assert gdn.chunk_plan(False, 4, 4096, 8, 256, 256, 64, torch.bfloat16) == "two_pass"
    o_ref, h_ref = _oracle_cached("head256", x)
    o, hT = _run(x, algo)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


# --- head size 256 on the tensor-core pair ----------------------------------------------------

def _w256(h0_std=0.02):
    return _workload("gdn", "bf16", 256, 256, 64, h0_std)


@pytest.mark.parametrize("B,T,H,h0", [(2, 333, 2, 0.02), (1, 64, 2, 0.02), (3, 5, 2, 0.0), (1, 1, 1, 0.02),
                                      (2, 4096 + 37, 8, 0.02)],
                         ids=["ragged", "one_chunk", "shorter_than_a_chunk", "one_token", "several_items_per_cta"])
def test_head256_tensor_core_pair(B, T, H, h0):
    x = W.chunk_inputs(_w256(h0), seed=21, B=B, T=T, H=H)
    assert _fits(x, "two_pass")
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "two_pass")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


def test_head256_more_state_ctas_than_sms():
    """90 chains, two state CTAs each (180 on 152 SMs): the state pass runs in two waves."""
    x = W.chunk_inputs(_w256(), seed=25, B=3, T=150, H=30)
    o_ref, h_ref = oracle_on_heads(x)
    o, hT = _run(x, "two_pass")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


def test_head256_packed_sequences_match_separate_runs_bitwise():
    lens = [130, 0, 64, 1, 200, 63, 65]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = W.chunk_inputs(_w256(), seed=22, B=1, T=int(cu[-1]), H=2)
    x["cu_seqlens"] = torch.from_numpy(cu)
    x["initial_state"] = torch.randn(len(lens), 2, 256, 256, generator=torch.Generator().manual_seed(3)) * 0.02
    o, hT = _run(x, "two_pass")
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        xn = {**x, "cu_seqlens": None, "initial_state": x["initial_state"][n:n + 1]}
        for key in ("q", "k", "v", "g", "beta"):
            xn[key] = x[key][:, a:b].contiguous()
        on, hn = _run(xn, "two_pass")
        assert np.array_equal(o[:, a:b], on), n
        assert np.array_equal(hT[n], hn[0]), n
    assert np.array_equal(hT[1], x["initial_state"][1].double().numpy())
    o_ref, h_ref = oracle_on_heads(x)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


def test_head256_bf16_output_and_no_final_state():
    # a bf16 o is the round-to-nearest-even of the same fp32 result; leaving out the final state changes nothing else
    x = W.chunk_inputs(_w256(), seed=23, B=2, T=150, H=2)
    o32, h32 = _run(x, "two_pass")
    o16, h16 = _run(x, "two_pass", o_dtype=torch.bfloat16)
    assert np.array_equal(o16, torch.from_numpy(o32).float().to(torch.bfloat16).double().numpy())
    assert np.array_equal(h16, h32)
    on, hn = _run(x, "two_pass", out_final=False)
    assert hn is None and np.array_equal(on, o32)


def test_head256_grouped_value_heads_and_activations():
    """H_v = 2 H_k at head size 256, with the gate and beta activated in the kernel: checked against the oracle on
    q, k repeated per value head and the oracle's own activations."""
    Hk, G = 2, 2
    x = W.chunk_inputs(_w256(), seed=24, B=2, T=200, H=Hk * G)
    gl, bl, A_log, dt_bias, g64, b64 = _raw_gates(x, 24)
    xr = dict(x)
    xr["q"] = x["q"][:, :, ::G].repeat_interleave(G, dim=2)
    xr["k"] = x["k"][:, :, ::G].repeat_interleave(G, dim=2)
    xr["g"], xr["beta"] = torch.from_numpy(g64), torch.from_numpy(b64)
    o_ref, h_ref = oracle_on_heads(xr)
    d = to_dev(x)
    o, hT = gdn.gdn_chunk_fwd(d["q"][:, :, ::G].contiguous(), d["k"][:, :, ::G].contiguous(), d["v"],
                              torch.from_numpy(gl).cuda(), torch.from_numpy(bl).cuda(), scale=x["scale"],
                              initial_state=d["initial_state"], output_final_state=True,
                              A_log=torch.from_numpy(A_log).cuda(), dt_bias=torch.from_numpy(dt_bias).cuda(),
                              beta_sigmoid=True, algo="two_pass")
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    assert_close(o.double().cpu().numpy(), o_ref, torch.bfloat16, "o")
    assert_close(hT.double().cpu().numpy(), h_ref, torch.bfloat16, "final state")


def _raw_gates(x, seed):
    """Raw gate and beta logits plus A_log, dt_bias per head, and the activated log alpha and beta the oracle takes,
    formed by the oracle's own pinned activations (oracle.gate_activation, oracle.beta_activation)."""
    rng = np.random.default_rng(seed)
    H = x["q"].shape[2]
    gl = rng.standard_normal(tuple(x["beta"].shape), dtype=np.float32)   # one gate logit per (token, head)
    bl = rng.standard_normal(tuple(x["beta"].shape), dtype=np.float32)
    A_log = np.log(rng.uniform(0.5, 16.0, size=H)).astype(np.float32)
    dt_bias = rng.normal(0.0, 0.1, size=H).astype(np.float32)
    return gl, bl, A_log, dt_bias, oracle.gate_activation(gl, A_log, dt_bias), oracle.beta_activation(bl)


def test_in_kernel_gate_and_beta_activation():
    x = W.chunk_inputs(W.config(1), seed=9, B=2, T=333, H=3)
    gl, bl, A_log, dt_bias, g64, b64 = _raw_gates(x, 9)
    xr = dict(x)
    xr["g"], xr["beta"] = torch.from_numpy(g64), torch.from_numpy(b64)   # the oracle sees the fp64 activation
    o_ref, h_ref = oracle_on_heads(xr)
    d = to_dev(x)
    o, hT = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], torch.from_numpy(gl).cuda(), torch.from_numpy(bl).cuda(),
                              scale=x["scale"], initial_state=d["initial_state"], output_final_state=True,
                              A_log=torch.from_numpy(A_log).cuda(), dt_bias=torch.from_numpy(dt_bias).cuda(),
                              beta_sigmoid=True)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    assert_close(o.double().cpu().numpy(), o_ref, torch.bfloat16, "o")
    assert_close(hT.double().cpu().numpy(), h_ref, torch.bfloat16, "final state")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_grouped_value_heads(kind):
    """H_v = 3 H_k: value head h reads q and k of key head h // 3 (checked against the oracle on q, k repeated
    per value head)."""
    Hk, G = 2, 3
    x = W.chunk_inputs(W.config(3 if kind == "kda" else 1), seed=10, B=2, T=200, H=Hk * G)
    xq = dict(x)
    xq["q"] = x["q"][:, :, ::G].contiguous()        # the key heads
    xq["k"] = x["k"][:, :, ::G].contiguous()
    xr = dict(x)
    xr["q"] = xq["q"].repeat_interleave(G, dim=2)  # what each value head sees
    xr["k"] = xq["k"].repeat_interleave(G, dim=2)
    o_ref, h_ref = oracle_on_heads(xr)
    o, hT = _run(xq, "auto")
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(hT, h_ref, torch.bfloat16, "final state")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_beta_in_zero_two_from_logits(kind):
    """beta = 2 sigmoid(b) in the kernel (negative eigenvalues of I - beta k k^T allowed); GDN also activates
    the gate from logits, KDA takes its per-channel gate as given."""
    x = W.chunk_inputs(W.config(3 if kind == "kda" else 1), seed=12, B=2, T=270, H=2)
    gl, bl, A_log, dt_bias, g64, b64 = _raw_gates(x, 12)
    xr = dict(x)
    xr["beta"] = torch.from_numpy(oracle.beta_activation(bl, 2))
    if kind == "gdn":
        xr["g"] = torch.from_numpy(g64)
    o_ref, h_ref = oracle_on_heads(xr)
    d = to_dev(x)
    bt = torch.from_numpy(bl).cuda()
    common = dict(scale=x["scale"], initial_state=d["initial_state"], output_final_state=True, beta_sigmoid=True,
                  allow_neg_eigval=True)
    if kind == "gdn":
        o, hT = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], torch.from_numpy(gl).cuda(), bt,
                                  A_log=torch.from_numpy(A_log).cuda(), dt_bias=torch.from_numpy(dt_bias).cuda(),
                                  **common)
    else:
        o, hT = gdn.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], bt, **common)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    assert_close(o.double().cpu().numpy(), o_ref, torch.bfloat16, "o")
    assert_close(hT.double().cpu().numpy(), h_ref, torch.bfloat16, "final state")


# --- the fp16 range of the tensor-core path ---------------------------------------------------

@pytest.mark.parametrize("kind", ["gdn", "kda", "gdn256"])
@pytest.mark.parametrize("v_scale", [1e2, 3e4, 1e6])
def test_fp16_range_limit_is_reported_never_silent(kind, v_scale):
    """The two-pass kernels round some intermediates to fp16 (largest finite value 65,504).  Values v scaled by up
    to 1e6, with beta near its upper bound 2 ("Gated Delta Network (GDN)", §5: beta in (0, 2)), either match the
    oracle or leave a non-finite value in o or the final state, which gdn_device_status reports as
    GDN_ERR_NONFINITE.  A non-finite output without that status is a failure."""
    w = W.HEAD256 if kind == "gdn256" else W.config(3 if kind == "kda" else 1)
    x = W.chunk_inputs(w, seed=14, B=1, T=256, H=2)
    x["v"] = (x["v"].float() * v_scale).to(torch.bfloat16)
    x["beta"] = torch.full_like(x["beta"], 1.95)
    d = to_dev(x)
    fn = gdn.kda_chunk_fwd if kind == "kda" else gdn.gdn_chunk_fwd
    o, hT = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["initial_state"],
               output_final_state=True, algo="two_pass")
    torch.cuda.synchronize()
    st = gdn.device_status()
    o, hT = o.double().cpu().numpy(), hT.double().cpu().numpy()
    all_finite = bool(np.isfinite(o).all() and np.isfinite(hT).all())
    if st == 5:                       # GDN_ERR_NONFINITE
        assert not all_finite
    else:
        assert st == 0 and all_finite
        o_ref, h_ref = oracle_on_heads(x)
        assert_close(o, o_ref, torch.bfloat16, "o")
        assert_close(hT, h_ref, torch.bfloat16, "final state")
    if v_scale >= 1e6:                # v itself is past the fp16 range: the status must say so
        assert st == 5


# --- bounded waits, ring depth and memory guards of the tensor-core path ------------------------

def _call(x, algo="two_pass", **kw):
    d = to_dev(x)
    fn = gdn.kda_chunk_fwd if x["gate_per_channel"] else gdn.gdn_chunk_fwd
    return fn(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["initial_state"],
              output_final_state=True, cu_seqlens=d["cu_seqlens"], chunk_size=x["chunk_size"], algo=algo, **kw)


@pytest.mark.parametrize("kind", ["gdn", "kda", "gdn256"])
def test_a_state_pass_wait_that_runs_out_is_reported_and_the_context_stays_usable(kind):
    """The test injection leaves out the state kernels' first record copy: their bounded waits give up (about 2 s
    each), the call reports GDN_ERR_TIMEOUT through gdn_device_status, the status clears, and the next call on the
    same context matches the oracle."""
    w = W.HEAD256 if kind == "gdn256" else W.config(3 if kind == "kda" else 1)
    x = W.chunk_inputs(w, seed=15, B=1, T=200, H=2)
    lib = gdn.load()
    gdn.device_status()                       # start from a clear status
    assert lib.gdn_test_inject(2) == 0        # GDN_TEST_FWD_RECORD_STALL
    _call(x)                                  # this call's outputs are unspecified
    torch.cuda.synchronize()
    assert gdn.device_status() == 4           # GDN_ERR_TIMEOUT, and cleared
    assert gdn.device_status() == 0
    o, hT = _run(x, "two_pass")
    o_ref, h_ref = oracle_on_heads(x)
    assert_close(o, o_ref, torch.bfloat16, "o after the timeout")
    assert_close(hT, h_ref, torch.bfloat16, "final state after the timeout")


@pytest.mark.parametrize("head", [128, 256])
def test_a_one_chunk_deep_ring_gives_bitwise_the_same_result(head):
    """The state kernel's two-stage ring run one chunk deep (test injection GDN_TEST_FWD_ONE_STAGE) changes only the
    timing of its copies and conversions against its products: packed ragged sequences give the same bits."""
    x = W.chunk_inputs(W.config(2), seed=16, T=3000, H=3)
    if head == 256:
        x = {**x, **{k: v for k, v in W.chunk_inputs(_w256(), seed=16, B=1, T=3000, H=3).items()
                     if k in ("q", "k", "v", "initial_state")}}
        x["initial_state"] = torch.randn(x["N"], 3, 256, 256, generator=torch.Generator().manual_seed(5)) * 0.02
    o1, h1 = _run(x, "two_pass")
    assert gdn.load().gdn_test_inject(3) == 0
    o2, h2 = _run(x, "two_pass")
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


GUARD = 4096          # bytes of guard before and after each buffer


def _guarded(shape, dtype, fill=0xA5):
    """A tensor of `shape` inside a larger byte buffer filled with `fill`; returns (view, buffer, offset, nbytes)."""
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((n + 2 * GUARD,), fill, dtype=torch.uint8, device="cuda")
    view = buf[GUARD:GUARD + n].view(dtype).view(shape)
    return view, buf, n


def _guards_intact(buf, n, fill=0xA5):
    host = buf.cpu()
    return bool((host[:GUARD] == fill).all()) and bool((host[GUARD + n:] == fill).all())


@pytest.mark.parametrize("case", ["gdn_ragged", "gdn_packed", "kda_ragged", "generic_f32", "gdn_bf16_o",
                                  "gdn256_packed"])
def test_guard_bytes_around_outputs_and_workspace_stay_untouched(case):
    """Host canaries: o, the final state and the caller workspace sit inside larger buffers whose guard bytes hold a
    sentinel; after the call every guard byte still holds it (no out-of-bounds store by a bulk copy, a tensor store
    or a partial tail chunk), and the result still matches the oracle."""
    if case == "gdn_packed":
        x = W.chunk_inputs(W.config(2), seed=17, T=1500, H=2)
    elif case == "gdn256_packed":
        x = W.chunk_inputs(W.config(2), seed=17, T=1500, H=2)
        x = {**x, **{k: v for k, v in W.chunk_inputs(_w256(), seed=17, B=1, T=1500, H=2).items()
                     if k in ("q", "k", "v")}}
        x["initial_state"] = torch.randn(x["N"], 2, 256, 256, generator=torch.Generator().manual_seed(6)) * 0.02
    elif case == "kda_ragged":
        x = W.chunk_inputs(W.config(3), seed=17, B=2, T=197, H=2)
    elif case == "generic_f32":
        x = W.chunk_inputs(W.config(0), seed=17, B=2, T=77, H=2)
    else:
        x = W.chunk_inputs(W.config(1), seed=17, B=2, T=333, H=3)
    B, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    N = x["N"]
    o_dtype = torch.bfloat16 if case == "gdn_bf16_o" else torch.float32
    o, ob, on = _guarded((B, T, H, dv), o_dtype)
    hT, hb, hn = _guarded((N, H, dk, dv), torch.float32)
    algo = "generic" if case == "generic_f32" else "two_pass"
    need = gdn.workspace_size(x["gate_per_channel"], B, T, H, dk, dv, x["chunk_size"], x["q"].dtype,
                              0 if x["cu_seqlens"] is None else N, algo, o_dtype)
    ws, wb, wn = _guarded((max(need, 1),), torch.uint8)
    _call(x, algo, o=o, final_state=hT, o_dtype=o_dtype, workspace=ws if need > 0 else None)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    assert _guards_intact(ob, on), "o guard bytes changed"
    assert _guards_intact(hb, hn), "final state guard bytes changed"
    assert _guards_intact(wb, wn), "workspace guard bytes changed"
    o_ref, h_ref = oracle_on_heads(x)
    tol = torch.float32 if case == "generic_f32" else torch.bfloat16
    if o_dtype == torch.float32:
        assert_close(o.double().cpu().numpy(), o_ref, tol, "o")
    else:   # a bf16 o is the round-to-nearest-even of the fp32 result (bf16 rounding alone exceeds the max bound)
        o32, _ = _call(x, algo)
        torch.cuda.synchronize()
        assert torch.equal(o.cpu(), o32.to(torch.bfloat16).cpu())
    assert_close(hT.double().cpu().numpy(), h_ref, tol, "final state")

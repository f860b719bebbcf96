"""The C-ABI library builds, loads and exports every entry point include/gdn.h declares.

Host-side argument checking is exercised too.  Every call here is rejected
before any CUDA work, so no GPU is needed and none is touched.
"""
import ctypes
import os
import re

import pytest

from gated_delta_rule_gdn_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _binding.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:gdn_status|const char\*)\s+(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_three_entry_points():
    names = _declared_functions()
    for n in ("gdn_chunk_fwd", "kda_chunk_fwd", "gdn_recurrent_step", "gdn_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_binding.lib_path())
    missing = [n for n in _declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_version(lib):
    assert b"sm_103a" in lib.gdn_version()


FAKE = 0x10000  # an aligned, never-dereferenced address: every call below fails validation first


def _chunk(lib, fn="gdn_chunk_fwd_algo", **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=1.0, h0=None, ofs=0, hT=None, cu=None, n=0, o=FAKE,
             B=1, T=64, H=1, dk=64, dv=64, C=64, dtype=1, odt=0, algo=0)
    a.update(kw)
    f = getattr(lib, fn)
    return f(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["ofs"], a["hT"], a["cu"], a["n"],
             a["o"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dtype"], a["odt"], a["algo"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(dk=0), 2), (dict(dv=257), 2), (dict(C=48), 2),
    (dict(C=128), 2), (dict(dtype=7), 1), (dict(q=None), 1), (dict(o=None), 1), (dict(ofs=1), 1),
    (dict(hT=FAKE), 1), (dict(cu=FAKE, B=2, n=2), 1), (dict(cu=FAKE, n=0), 1), (dict(q=FAKE + 1), 1),
    (dict(scale=float("nan")), 1), (dict(algo=9), 1), (dict(odt=3), 1), (dict(o=FAKE + 2), 1), (dict(algo=2, dtype=0), 2), (dict(algo=2, dk=64, dv=32), 2),
])
def test_chunk_argument_checks(lib, kw, status):
    assert _chunk(lib, **kw) == status
    assert _binding.last_error()
    assert _chunk(lib, fn="kda_chunk_fwd_algo", **kw) == status


def test_step_argument_checks(lib):
    f = lib.gdn_recurrent_step
    ok = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, b=FAKE, s=1.0, st=FAKE, o=FAKE, N=4, H=2, dk=128, dv=128, dt=1, odt=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["g"], a["b"], a["s"], a["st"], a["o"], a["N"], a["H"], a["dk"], a["dv"],
                 a["dt"], a["odt"], None)
    assert call(N=0) == 1
    assert call(st=None) == 1
    assert call(dk=257) == 2
    assert call(dt=5) == 1
    assert call(q=FAKE + 2, dt=0) == 1
    assert call(s=float("inf")) == 1
    assert call(odt=2) == 1
    assert call(o=FAKE + 2) == 1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import gated_delta_rule_gdn_gb300 as gdn
    x = torch.zeros(1, 4, 1, 8)
    with pytest.raises(ValueError):
        gdn.gdn_chunk_fwd(x, x, x, torch.zeros(1, 4, 1), torch.zeros(1, 4, 1))


def test_plan_and_workspace_sizes(lib):
    import torch
    bf = torch.bfloat16
    # the prefill shape resolves to the two-pass tcgen05 path; fp32 and small heads to the generic kernel
    assert _binding.chunk_plan(False, 4, 4096, 16, 128, 128, 64, bf) == "two_pass"
    assert _binding.chunk_plan(True, 2, 8192, 32, 128, 128, 64, bf) == "two_pass"
    assert _binding.chunk_plan(False, 1, 64, 1, 16, 16, 16, torch.float32) == "generic"
    with pytest.raises(_binding.GdnError) as err:      # the retired single-launch kernel is refused
        _binding.chunk_plan(False, 4, 4096, 16, 128, 128, 64, bf, algo="tcgen05")
    assert err.value.status == 2 and "retired" in str(err.value)
    # per (chunk slot, head): 32,768 bytes for the scalar gate, 74,240 for the per-channel gate;
    # floor(B T / 64) + N + 1 slots
    assert _binding.workspace_size(False, 4, 4096, 16, 128, 128, 64, bf) == (256 + 4 + 1) * 16 * 32768
    assert _binding.workspace_size(False, 1, 65536, 32, 128, 128, 64, bf, n_seqs=8) == (1024 + 8 + 1) * 32 * 32768
    assert _binding.workspace_size(True, 2, 8192, 32, 128, 128, 64, bf) == (256 + 2 + 1) * 32 * 74240
    assert _binding.workspace_size(False, 1, 64, 1, 16, 16, 16, torch.float32) == 0
    with pytest.raises(_binding.GdnError):
        _binding.workspace_size(False, 1, 64, 1, 64, 64, 64, bf, algo="two_pass")


def _chunk_ws(lib, ws, ws_bytes, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=1.0, h0=None, ofs=0, hT=None, cu=None, n=0, o=FAKE,
             B=1, T=64, H=1, dk=128, dv=128, C=64, dtype=1, odt=0, algo=3)
    a.update(kw)
    return lib.gdn_chunk_fwd_ws(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["ofs"], a["hT"],
                                a["cu"], a["n"], a["o"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dtype"],
                                a["odt"], a["algo"], ws, ws_bytes, None)


def test_workspace_argument_checks(lib):
    need = (1 + 1 + 1) * 1 * 32768
    assert _chunk_ws(lib, FAKE, need - 16) == 1            # too small
    assert "workspace" in _binding.last_error()
    assert _chunk_ws(lib, FAKE + 16, need) == 1            # not 256-byte aligned
    assert _chunk_ws(lib, FAKE, need, dk=64, dv=64) == 2   # the two-pass kernels need d = 128


def test_gate_activation_argument_checks(lib):
    act = _binding.GateAct(FAKE, None, 1)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, None, 0, None, None, 0, FAKE, 1, 64, 1, 128, 128, 64, 1, 0]
    # the fp32 inputs below resolve to the generic kernel, which has no activation: refused before any launch
    a32 = list(args)
    a32[18] = 0
    assert lib.gdn_chunk_fwd_act(*a32, ctypes.byref(act), 0, None, 0, None) == 2
    assert "two-pass" in _binding.last_error()
    bad = _binding.GateAct(None, FAKE, 0)        # dt_bias without A_log
    assert lib.gdn_chunk_fwd_act(*args, ctypes.byref(bad), 0, None, 0, None) == 1
    odd = _binding.GateAct(FAKE + 2, None, 0)    # misaligned A_log
    assert lib.gdn_chunk_fwd_act(*args, ctypes.byref(odd), 0, None, 0, None) == 1


def test_grouped_value_head_argument_checks(lib):
    # gdn_chunk_fwd_ex: per_channel, then the chunk arguments with H_k before H_v
    def chunk(Hk, Hv, dtype=1, algo=0):
        return lib.gdn_chunk_fwd_ex(0, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, None, 0, None, None, 0, FAKE, 1, 64, Hk, Hv,
                                    128, 128, 64, dtype, 0, None, algo, None, 0, None)
    assert chunk(2, 5) == 1                      # H_v not a multiple of H_k
    assert "key heads" in _binding.last_error()
    assert chunk(-1, 4) == 1
    assert chunk(2, 4, algo=2) == 2              # the fused single-kernel path reads one key head per value head
    assert chunk(2, 4, dtype=0) == 2             # fp32 resolves to the generic kernel: refused before any launch

    def step(Hk, Hv):
        return lib.gdn_recurrent_step_ex(0, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, FAKE, 4, Hk, Hv, 128, 128, 1, 0,
                                         None, None)
    assert step(3, 4) == 1
    assert "key heads" in _binding.last_error()


def test_beta_activation_mode_checks(lib):
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, None, 0, None, None, 0, FAKE, 1, 64, 1, 128, 128, 64, 1, 0]
    three = _binding.GateAct(None, None, 3)
    assert lib.gdn_chunk_fwd_act(*args, ctypes.byref(three), 0, None, 0, None) == 1
    assert "beta_sigmoid" in _binding.last_error()
    # the per-channel entries take the beta activation but not the gate activation
    gate = _binding.GateAct(FAKE, None, 0)
    assert lib.gdn_recurrent_step_ex(1, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, FAKE, 4, 2, 2, 128, 128, 1, 0,
                                     ctypes.byref(gate), None) == 2
    assert "scalar gate" in _binding.last_error()


@pytest.mark.parametrize("per_channel, dk, dv, C, dtype, varlen, expect", [
    # the tensor-core pairs: bf16, chunk 64, d_k = d_v = 128 (either gate) or 256 (scalar gate), packed or not
    (False, 128, 128, 64, "bf16", False, "two_pass"),
    (False, 128, 128, 64, "bf16", True, "two_pass"),
    (True, 128, 128, 64, "bf16", False, "two_pass"),
    (False, 256, 256, 64, "bf16", False, "two_pass"),
    (False, 256, 256, 64, "bf16", True, "two_pass"),
    # everything else on the generic kernel
    (True, 256, 256, 32, "bf16", False, "generic"),
    (False, 256, 128, 64, "bf16", False, "generic"),
    (False, 128, 256, 64, "bf16", False, "generic"),
    (False, 192, 192, 64, "bf16", False, "generic"),
    (False, 64, 64, 64, "bf16", False, "generic"),
    (False, 128, 128, 32, "bf16", False, "generic"),
    (False, 128, 128, 64, "f32", False, "generic"),
    (False, 256, 256, 64, "f32", False, "generic"),
    (True, 128, 128, 64, "f32", False, "generic"),
])
def test_auto_dispatch_table(lib, per_channel, dk, dv, C, dtype, varlen, expect):
    # which kernel the default (auto) request resolves to, for the shapes the documentation lists
    import torch
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    assert _binding.chunk_plan(per_channel, 1, 300, 2, dk, dv, C, dt, varlen) == expect


def test_head_sizes_up_to_256_and_the_generic_kernels_shared_memory(lib):
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    # d_k = d_v = 256 in bf16 with the scalar gate and chunk 64 has its tensor-core pair; other head sizes above 128
    # run on the generic kernel: chunk 64 for the scalar gate ...
    assert _binding.chunk_plan(False, 1, 300, 2, 256, 256, 64, bf) == "two_pass"
    assert _binding.chunk_plan(False, 1, 300, 2, 256, 256, 64, bf, algo="generic") == "generic"
    assert _binding.chunk_plan(False, 1, 300, 2, 256, 128, 64, bf) == "generic"
    assert _binding.chunk_plan(False, 1, 300, 2, 256, 64, 64, f32) == "generic"
    # the head-256 pair's workspace: (floor(B T / 64) + N + 1) slots x H records of 114,688 bytes ([-W; Q~] 64 KB,
    # K~ 32 KB, P^T and T diag(beta) 8 KB each); the d = 128 pair's records are 32,768 bytes
    assert _binding.workspace_size(False, 2, 4096, 8, 256, 256, 64, bf) == (128 + 2 + 1) * 8 * 114_688
    assert _binding.workspace_size(False, 2, 4096, 8, 128, 128, 64, bf) == (128 + 2 + 1) * 8 * 32_768
    # ... chunk 32 or less for the per-channel gate; chunk 64 would not fit one CTA's shared memory
    assert _binding.chunk_plan(True, 1, 300, 2, 256, 256, 32, bf) == "generic"
    with pytest.raises(_binding.GdnError) as e:
        _binding.chunk_plan(True, 1, 300, 2, 256, 256, 64, bf)
    assert "shared memory" in str(e.value) and "chunk_size" in str(e.value)
    # the same refusal from a forward call, before any launch (fake pointers are never touched)
    assert _chunk(lib, fn="kda_chunk_fwd_algo", dk=256, dv=256, C=64) == 2
    assert "shared memory" in _binding.last_error()
    with pytest.raises(_binding.GdnError):
        _binding.chunk_plan(False, 1, 300, 2, 257, 64, 64, bf)


def _bwd(lib, **kw):
    a = dict(pc=0, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=1.0, h0=None, do=FAKE, dhT=None, cu=None, n=0,
             gq=FAKE, gk=FAKE, gv=FAKE, gg=FAKE, gb=FAKE, gh0=None, B=1, T=64, H=1, dk=64, dv=64, C=0, dtype=1,
             dodt=1, ws=FAKE, wsb=16)
    a.update(kw)
    return lib.gdn_chunk_bwd(a["pc"], a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["do"],
                             a["dhT"], a["cu"], a["n"], a["gq"], a["gk"], a["gv"], a["gg"], a["gb"], a["gh0"], a["B"],
                             a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dtype"], a["dodt"], a["ws"], a["wsb"], None)


# The default arguments above carry a 16-byte workspace, too small for any request, so each call fails its
# checks before a launch even where the case under test would pass.
@pytest.mark.parametrize("kw,status", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(dk=0), 2), (dict(dv=257), 2), (dict(dk=257), 2),
    (dict(C=48), 2), (dict(C=64), 2), (dict(pc=1, dk=256, C=32), 2), (dict(dtype=7), 1), (dict(dodt=5), 1),
    (dict(q=None), 1), (dict(do=None), 1), (dict(gq=None), 1), (dict(gg=None), 1), (dict(gb=None), 1),
    (dict(do=FAKE + 1), 1), (dict(gq=FAKE + 2), 1), (dict(gh0=FAKE + 2), 1), (dict(h0=FAKE + 1), 1),
    (dict(scale=float("nan")), 1), (dict(cu=FAKE, B=2, n=2), 1), (dict(cu=FAKE, n=0), 1), (dict(cu=FAKE + 1, n=1), 1),
    (dict(), 1), (dict(ws=FAKE + 16, wsb=1 << 40), 1),
])
def test_backward_argument_checks(lib, kw, status):
    assert _bwd(lib, **kw) == status
    assert _binding.last_error()
    if "pc" not in kw:
        assert _bwd(lib, pc=1, **kw) == status


def test_backward_workspace_sizes(lib):
    # per (chunk slot, head): the entry state and the gradient of h_out (fp32 [d_k, d_v] each); Delta, Y and Z
    # (fp32 [C, d_v] each); a per-chunk record of the state-independent products; then room for the activated gate
    # and beta ([B, T, H] each).  So the size is affine in the number of slots and above the states and tiles alone.
    # The default chunk is 16.
    def floor_bytes(slots, H, dk, dv, C):
        return slots * H * (2 * dk * dv + 3 * C * dv) * 4
    size = lambda *a: _binding.bwd_workspace_size(*a)
    s1 = size(False, 4, 4096, 16, 128, 128)              # chunk 16: 4 x 257 slots
    assert s1 == size(False, 4, 4096, 16, 128, 128, 16)
    s2 = size(False, 8, 4096, 16, 128, 128)              # twice the slots
    assert s2 == 2 * s1 and s1 > floor_bytes(4 * 257, 16, 128, 128, 16)
    s32 = size(False, 4, 4096, 16, 128, 128, 32)         # chunk 32: 4 x 129 slots
    assert s32 > floor_bytes(4 * 129, 16, 128, 128, 32)
    sv = size(True, 1, 65536, 32, 128, 128, 0, 8)        # packed: floor(T / C) + 2 n_seqs slots
    assert sv > floor_bytes(65536 // 16 + 16, 32, 128, 128, 16)
    # affine in the packed slot count floor(T / C) + 2 n_seqs (plus the fixed room for the activated gate and beta)
    s16, s24 = size(True, 1, 65536, 32, 128, 128, 0, 16), size(True, 1, 65536, 32, 128, 128, 0, 24)
    assert s24 - s16 == s16 - sv > 0
    assert size(False, 2, 0, 3, 64, 32) > 0
    # d_k = 256 with the per-channel gate: chunk 32 does not fit one CTA
    assert size(True, 1, 100, 2, 256, 128) == size(True, 1, 100, 2, 256, 128, 16)
    with pytest.raises(_binding.GdnError, match="shared memory"):
        size(True, 1, 100, 2, 256, 128, 32)


def test_test_injection_argument_checks(lib):
    assert lib.gdn_test_inject(7) == 1
    assert lib.gdn_test_inject(-1) == 1
    for what in (1, 2, 3):       # backward record stall, forward record stall, one-chunk-deep forward ring
        assert lib.gdn_test_inject(what) == 0
    assert lib.gdn_test_inject(0) == 0


def test_backward_activation_argument_checks(lib):
    import ctypes as ct

    def call(act, gA=FAKE, gdt=None, pc=0):
        return lib.gdn_chunk_bwd_act(pc, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, FAKE, None, None, 0, FAKE, FAKE,
                                     FAKE, FAKE, FAKE, None, gA, gdt, 1, 64, 1, 64, 64, 0, 1, 1, act, FAKE, 16, None)
    act = _binding.GateAct(FAKE, None, 0)
    assert call(ct.byref(act), gA=None) == 1                      # A_log needs grad_A_log
    assert call(ct.byref(act), gdt=FAKE) == 1                     # grad_dt_bias needs dt_bias
    assert call(ct.byref(act), pc=1) == 2                         # the gate activation is scalar-gate only
    bad = _binding.GateAct(None, None, 3)
    assert call(ct.byref(bad)) == 1                               # beta_sigmoid 0..2
    ok = _binding.GateAct(FAKE, FAKE, 1)
    assert call(ct.byref(ok), gdt=FAKE) == 1                      # all valid but the 16-byte workspace: no launch

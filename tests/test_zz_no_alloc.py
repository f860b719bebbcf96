"""gdn_chunk_fwd_noalloc: the two-pass chunk forward with the library's static scratch.

Collected last (file name), and independent of every other test file: it passes
alone and after the rest.  The GPU tests check consecutive calls against the
caller-workspace entry point bit for bit, including a small packed call made
after a large one has left other data in the scratch; the CPU tests check that
requests above the 64 MiB scratch are refused before anything is launched, at
the exact capacity boundary of each gate form.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_gdn_gb300 as gdn
from gated_delta_rule_gdn_gb300 import _binding, build, workloads as W

SCRATCH_BYTES = 64 << 20
FAKE = 0x10000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def _need(per_channel, B, T, H, n_seqs=0, d=128):
    return _binding.workspace_size(per_channel, B, T, H, d, d, 64, torch.bfloat16, n_seqs=n_seqs)


def _noalloc_fake(lib, per_channel, B, T, H, d=128):
    return lib.gdn_chunk_fwd_noalloc(int(per_channel), FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, None, 0, None, None, 0,
                                     FAKE, B, T, H, d, d, 64, 1, 0, None)


def test_oversized_request_is_refused_before_any_launch(lib):
    B, T, H = 4, 4096, 16          # (256 + 4 + 1) * 16 records of 32,768 bytes > 64 MiB
    assert _need(False, B, T, H) > SCRATCH_BYTES
    assert _noalloc_fake(lib, False, B, T, H) == 2
    msg = _binding.last_error()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg


@pytest.mark.parametrize("per_channel, d, H_fit", [(False, 128, 31), (True, 128, 13), (False, 256, 8)])
def test_capacity_boundary(lib, per_channel, d, H_fit):
    """One 4096-token sequence has 4096 / 64 + 2 = 66 slots: the largest head count whose records fit the scratch
    is accepted by the size check, one more head is refused (the head-256 record is 112 KB: 8 heads x 66 slots)."""
    T = 4096
    assert _need(per_channel, 1, T, H_fit, d=d) <= SCRATCH_BYTES < _need(per_channel, 1, T, H_fit + 1, d=d)
    assert _noalloc_fake(lib, per_channel, 1, T, H_fit + 1, d) == 2
    assert "scratch" in _binding.last_error()


def _inputs(kind, seed, T, H, packed=False):
    cfg = W.HEAD256 if kind == "gdn256" else W.config(2 if packed else (3 if kind == "kda" else 1))
    x = W.chunk_inputs(cfg, seed=seed, B=1, T=T, H=H)
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}, kind == "kda"


def _ref(x, per_channel):
    fn = gdn.kda_chunk_fwd if per_channel else gdn.gdn_chunk_fwd
    o, h = fn(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"], initial_state=x["initial_state"],
              output_final_state=True, cu_seqlens=x["cu_seqlens"], algo="two_pass")
    return o, h


def _noalloc(x, pc):
    return gdn.chunk_fwd_noalloc(pc, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"],
                                 initial_state=x["initial_state"], output_final_state=True,
                                 cu_seqlens=x["cu_seqlens"])


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["gdn", "kda", "gdn256"])
def test_two_consecutive_calls_match_the_workspace_entry_point(lib, kind):
    T, H = 1000, 4                  # (15 + 1 + 1) * 4 records: well inside the scratch
    xa, pc = _inputs(kind, 11, T, H)
    xb, _ = _inputs(kind, 12, T, H)
    outs = [_noalloc(x, pc) for x in (xa, xb)]   # the second call reuses the scratch the first one wrote
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    for (o, h), x in zip(outs, (xa, xb)):
        o_ref, h_ref = _ref(x, pc)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(h, h_ref)
    assert not torch.equal(outs[0][0], outs[1][0])


@pytest.mark.gpu
@pytest.mark.parametrize("kind, H", [("gdn", 31), ("kda", 13)])
def test_largest_request_that_fits(lib, kind, H):
    T = 4096
    x, pc = _inputs(kind, 13, T, H)
    assert _need(pc, 1, T, H) <= SCRATCH_BYTES
    o, h = _noalloc(x, pc)
    o_ref, h_ref = _ref(x, pc)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_small_packed_call_after_a_large_one(lib, kind):
    """Nothing in the scratch needs to start at zero: a large call fills it, then a small packed call with short
    sequences (whose records sit where the large call left other data) still matches the workspace entry point."""
    big, pc = _inputs(kind, 21, 4096, 12)
    _noalloc(big, pc)
    small, _ = _inputs(kind, 22, 300, 3, packed=True)
    if pc:   # the packed recipe draws a scalar gate; give the per-channel form a per-channel gate of the same size
        small["g"] = small["g"][..., None].expand(*small["g"].shape, 128).contiguous()
    o, h = _noalloc(small, pc)
    o_ref, h_ref = _ref(small, pc)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)
